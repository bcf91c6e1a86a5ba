// Host side of the shared-prefix decode: which sequences of a batch read the
// same leading pages, and how many tokens of them they share.
//
// "mlx-paged-attention", feature 2 and "PagedAttention原理" §3.3.3: forked
// sequences (parallel samples, beams) hold their parent's pages until they
// write to them, so their block tables begin with the same physical pages.
// Runs of consecutive sequences whose first page is the same form a group;
// its shared length is the common run of leading pages, cut to whole pages
// below the shortest member's length (every member keeps at least one token of
// its own).  Sequences that share nothing with a neighbour are gathered into
// groups of shared length 0.
#include <algorithm>
#include <cstdint>

#include "../../include/pa.h"

extern "C" {

int pa_cascade_groups(const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                      int max_blocks_per_seq, int block_size, int32_t* group_start,
                      int32_t* shared_lens, int* num_groups) {
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || !num_groups)
    return PA_ERR_INVALID_ARG;
  *num_groups = 0;
  if (num_seqs == 0) {
    if (group_start) group_start[0] = 0;
    return PA_OK;
  }
  if (!block_tables || !context_lens || !group_start || !shared_lens) return PA_ERR_INVALID_ARG;
  auto table = [&](int b) { return block_tables + static_cast<int64_t>(b) * max_blocks_per_seq; };
  auto pages_of = [&](int b) {
    const int64_t L = context_lens[b];
    return static_cast<int>(std::min<int64_t>((L + block_size - 1) / block_size, max_blocks_per_seq));
  };
  int g = 0;
  bool open_plain = false;                  // the last group shares nothing: extend it
  int i = 0;
  while (i < num_seqs) {
    if (context_lens[i] < 0) return PA_ERR_INVALID_ARG;
    int j = i + 1;
    int common = pages_of(i);
    int64_t min_len = context_lens[i];
    const int32_t first = table(i)[0];
    while (common > 0 && first >= 0 && j < num_seqs && context_lens[j] > 0 &&
           table(j)[0] == first) {
      int k = 0;
      const int lim = std::min(common, pages_of(j));
      while (k < lim && table(j)[k] == table(i)[k]) ++k;
      common = k;
      min_len = std::min<int64_t>(min_len, context_lens[j]);
      ++j;
    }
    const int64_t below = min_len > 0 ? (min_len - 1) / block_size : 0;
    const int64_t shared = std::min<int64_t>(common, below) * block_size;
    if (j - i >= 2 && shared > 0) {
      group_start[g] = i;
      shared_lens[g] = static_cast<int32_t>(shared);
      ++g;
      open_plain = false;
      i = j;
      continue;
    }
    if (!open_plain) {
      group_start[g] = i;
      shared_lens[g] = 0;
      ++g;
      open_plain = true;
    }
    ++i;
  }
  group_start[g] = num_seqs;
  *num_groups = g;
  return PA_OK;
}

}  // extern "C"
