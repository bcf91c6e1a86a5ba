"""Reference block manager -- test infrastructure only.

Written from "PagedAttention原理" (vLLM long-sequence memory guide, ch. 3):
  * §3.3.2 (allocation and release): a request starts with one page; on each new
    token, if its current page is full a page is taken from the free list and the
    page table is extended; when the request ends its physical pages go back to
    the free list.
  * §3.3.4 (teaching code): the free list is a Python list used as a stack --
    pages are taken with ``pop()`` from its end and returned with ``append`` in
    page-table order; an empty free list is an out-of-memory error.
  * §3.3.3 (shared pages) and the pitfall note after §3.3.4: pages shared by
    several requests (beam search, parallel sampling, a common prompt) carry a
    reference count and only return to the free list when it reaches zero.
and from "mlx-paged-attention", feature 2: a shared page is copied only when a
holder is about to modify it (copy-on-write); and from "PagedAttention MLX：为Apple
Silicon打造的高吞吐量LLM推理引擎" (feature list, dynamic scheduling; architecture,
physical KV pool): the pages of an inactive request can be swapped out to CPU
memory and back.

Readings where the pages are silent (each listed in the design notes):
  * fork(parent, child) gives the child the parent's page table and length and
    adds one reference to each page;
  * a writer whose target page has refcount > 1 takes a fresh page, copies, and
    drops one reference from the old page; the last holder (refcount 1) writes in
    place;
  * a failed allocation leaves every piece of state unchanged;
  * swapping moves a whole sequence: swap_out gives each of its pages (in table
    order) a host block from a LIFO host free list and drops the device
    reference (pages reaching zero return to the device free list, table order);
    swap_in gives each host block a device page from the device free list and
    returns the host blocks (table order).  A swapped sequence keeps its length;
    it cannot grow or be forked until it is swapped in; free releases its host
    blocks.  A page still shared with a resident sequence stays on the device
    for that holder; the swapped copy is private from then on.
"""
from __future__ import annotations


class OutOfBlocks(RuntimeError):
    """The free list is empty (the teaching code's out-of-memory error)."""


class Swapped(RuntimeError):
    """The sequence's pages are in host memory."""


class RefBlockManager:
    def __init__(self, num_blocks: int, block_size: int, initial_free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.block_size = int(block_size)
        self.num_blocks = int(num_blocks)
        if initial_free_order is None:
            self.free_pages = list(range(num_blocks))
        else:
            self.free_pages = [int(x) for x in initial_free_order]
            if sorted(self.free_pages) != list(range(num_blocks)):
                raise ValueError("initial free order must be a permutation of the pool")
        self.refcount = [0] * num_blocks
        self.page_tables: dict[int, list[int]] = {}
        self.lengths: dict[int, int] = {}
        self.host_free: list[int] = []
        self.swapped: dict[int, list[int]] = {}       # sequence -> its host blocks

    # -- allocation -------------------------------------------------------
    def _take_page(self) -> int:
        if not self.free_pages:
            raise OutOfBlocks("no free page")
        page = self.free_pages.pop()
        self.refcount[page] = 1
        return page

    def _resident(self, seq_id: int) -> list:
        if seq_id in self.swapped:
            raise Swapped(f"sequence {seq_id} is swapped out")
        return self.page_tables[seq_id]

    def add_seq(self, seq_id: int) -> None:
        """A new request gets its first page right away (§3.3.2 first step)."""
        if seq_id in self.page_tables or seq_id in self.swapped:
            raise KeyError(f"sequence {seq_id} exists")
        page = self._take_page()
        self.page_tables[seq_id] = [page]
        self.lengths[seq_id] = 0

    def append_slot(self, seq_id: int):
        """Reserve the slot of the sequence's next token.

        Returns (slot, cow_src, cow_dst); cow_* are -1 when no copy is needed.
        """
        table = self._resident(seq_id)
        length = self.lengths[seq_id]
        index, offset = divmod(length, self.block_size)
        if index == len(table):
            # the last page is full: take a new one and extend the table
            page = self._take_page()
            table.append(page)
            self.lengths[seq_id] = length + 1
            return page * self.block_size + offset, -1, -1
        page = table[index]
        if self.refcount[page] > 1:
            # shared page about to be modified: copy it first
            fresh = self._take_page()
            self.refcount[page] -= 1
            table[index] = fresh
            self.lengths[seq_id] = length + 1
            return fresh * self.block_size + offset, page, fresh
        self.lengths[seq_id] = length + 1
        return page * self.block_size + offset, -1, -1

    def fork(self, parent: int, child: int) -> None:
        if child in self.page_tables or child in self.swapped:
            raise KeyError(f"sequence {child} exists")
        table = self._resident(parent)
        for page in table:
            self.refcount[page] += 1
        self.page_tables[child] = list(table)
        self.lengths[child] = self.lengths[parent]

    def free(self, seq_id: int) -> None:
        """Drop one reference per page; pages reaching zero go back in table order.
        A swapped sequence returns its host blocks instead."""
        if seq_id in self.swapped:
            self.host_free.extend(self.swapped.pop(seq_id))
            del self.lengths[seq_id]
            return
        table = self.page_tables.pop(seq_id)
        del self.lengths[seq_id]
        for page in table:
            self.refcount[page] -= 1
            if self.refcount[page] == 0:
                self.free_pages.append(page)

    # -- swapping to host memory ------------------------------------------
    def enable_swap(self, num_host_blocks: int, initial_host_order=None) -> None:
        if num_host_blocks <= 0:
            raise ValueError("num_host_blocks must be positive")
        if initial_host_order is None:
            self.host_free = list(range(num_host_blocks))
        else:
            self.host_free = [int(x) for x in initial_host_order]
            if sorted(self.host_free) != list(range(num_host_blocks)):
                raise ValueError("initial host order must be a permutation of the host pool")
        self.num_host_blocks = int(num_host_blocks)

    def swap_out(self, seq_id: int):
        """Returns the copies to run, [(device page, host block)], in table order."""
        table = self._resident(seq_id)
        if len(self.host_free) < len(table):
            raise OutOfBlocks("no free host block")
        host = [self.host_free.pop() for _ in table]
        for page in table:
            self.refcount[page] -= 1
            if self.refcount[page] == 0:
                self.free_pages.append(page)
        del self.page_tables[seq_id]
        self.swapped[seq_id] = host
        return list(zip(table, host))

    def swap_in(self, seq_id: int):
        """Returns the copies to run, [(host block, device page)], in table order."""
        host = self.swapped[seq_id]
        if len(self.free_pages) < len(host):
            raise OutOfBlocks("no free page")
        table = [self._take_page() for _ in host]
        self.host_free.extend(host)
        del self.swapped[seq_id]
        self.page_tables[seq_id] = table
        return list(zip(host, table))

    def host_free_list(self):
        return list(self.host_free)

    # -- queries ----------------------------------------------------------
    def block_table(self, seq_id: int):
        return list(self._resident(seq_id)), self.lengths[seq_id]

    def num_free(self) -> int:
        return len(self.free_pages)

    def free_list(self):
        return list(self.free_pages)

    def stats(self):
        """(used pages, free pages, pages with refcount > 1, internal waste in token slots).

        Waste counts unused slots of the pages each sequence holds, one sequence at
        a time: sum over sequences of (pages * block_size - length).
        """
        used = sum(1 for r in self.refcount if r > 0)
        shared = sum(1 for r in self.refcount if r > 1)
        waste = sum(len(t) * self.block_size - self.lengths[s] for s, t in self.page_tables.items())
        return used, len(self.free_pages), shared, waste
