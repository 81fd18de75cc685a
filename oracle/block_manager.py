"""Oracle for the host-side paged block manager. Test infrastructure only.

Follows "KV Cache + Speculative Decoding" section 6.2 (the PagedKVCache
sketch: a free list used as a stack, one reference count per physical page,
a block table per request; allocate, append_token with copy-on-write, free,
share_prefix over whole pages) and the fork of "KV Cache" section 3.3
(PagedAttention: the new request's table is a copy of the source's, every
page's count goes up by one). Rollback after verification follows section 7
of the first page (the cache must end each round holding every token of the
sequence but the last; production engines roll back by editing the block
table).

Readings where the pages leave a step open:
  - A sequence also records its length in tokens; allocate(n_tokens) sets it,
    and the table always holds exactly ceil(len / page_size) pages.
  - extend(seq_ids, n_new) runs the page logic of append_token for the
    positions len .. len+n_new-1 of each sequence in turn (sequence order,
    then position order) without writing K/V: a position past the table
    pops a fresh page; a position on a page whose count is above one pops a
    fresh page, moves one reference to it, and records (old, new) so the
    caller can copy the page's contents on the device. Unlike the sketch's
    bare pop, the batch is all-or-nothing: if the free list is too short
    for the whole batch, nothing changes.
  - share_prefix(src, dst, n) gives dst the first n // page_size pages of src
    and the length (n // page_size) * page_size.
  - truncate(seq, new_len) keeps the first ceil(new_len / page_size) pages and
    releases the rest in table order, each like free() does (count down, back
    on the free list at zero).
  - commit_verify: after a round that appended n_new = K+1 rows and accepted
    num_accepted drafts, the cache keeps every row but the rejected ones and
    the not-yet-cached emitted token: len - n_new + num_accepted + 1.
"""


class OutOfBlocks(Exception):
    pass


class PagedBlockManager:
    def __init__(self, num_blocks, page_size=16):
        if num_blocks < 1 or page_size < 1:
            raise ValueError("num_blocks and page_size must be positive")
        self.page_size = page_size
        self.free_list = list(range(num_blocks))
        self.ref_count = [0] * num_blocks
        self.block_table = {}
        self.length = {}

    # -- helpers -----------------------------------------------------------
    def _pages_for(self, n_tokens):
        return (n_tokens + self.page_size - 1) // self.page_size

    def _release(self, pid):
        self.ref_count[pid] -= 1
        if self.ref_count[pid] == 0:
            self.free_list.append(pid)

    def _need_new(self, seq_id):
        if seq_id in self.block_table:
            raise KeyError("sequence %r already exists" % (seq_id,))

    # -- section 6.2 operations -------------------------------------------
    def allocate(self, seq_id, n_tokens):
        self._need_new(seq_id)
        if n_tokens < 0:
            raise ValueError("n_tokens < 0")
        n = self._pages_for(n_tokens)
        if len(self.free_list) < n:
            raise OutOfBlocks()
        pages = [self.free_list.pop() for _ in range(n)]
        for pid in pages:
            self.ref_count[pid] = 1
        self.block_table[seq_id] = pages
        self.length[seq_id] = n_tokens

    def free(self, seq_id):
        for pid in self.block_table[seq_id]:
            self._release(pid)
        del self.block_table[seq_id]
        del self.length[seq_id]

    def share_prefix(self, src, dst, n_tokens):
        self._need_new(dst)
        if n_tokens < 0 or n_tokens > self.length[src]:
            raise ValueError("n_tokens outside [0, len(src)]")
        n = n_tokens // self.page_size
        prefix = self.block_table[src][:n]
        for pid in prefix:
            self.ref_count[pid] += 1
        self.block_table[dst] = list(prefix)
        self.length[dst] = n * self.page_size

    def fork(self, src, dst):
        self._need_new(dst)
        pages = list(self.block_table[src])
        for pid in pages:
            self.ref_count[pid] += 1
        self.block_table[dst] = pages
        self.length[dst] = self.length[src]

    def _pages_needed(self, seq_ids, n_new):
        """Free pages the extend of this batch pops (a dry run of its counts)."""
        extra = {}
        need = 0
        for s in seq_ids:
            table = self.block_table[s]
            L = self.length[s]
            last = None
            for pos in range(L, L + n_new):
                idx = pos // self.page_size
                if idx == last:
                    continue
                last = idx
                if idx >= len(table):
                    need += 1
                    continue
                pid = table[idx]
                if self.ref_count[pid] + extra.get(pid, 0) > 1:
                    need += 1
                    extra[pid] = extra.get(pid, 0) - 1
        return need

    def extend(self, seq_ids, n_new):
        """Make positions len .. len+n_new-1 of every sequence writable.

        Returns the copy-on-write pairs [(src_page, dst_page), ...] in the
        order they were made.
        """
        if n_new < 0:
            raise ValueError("n_new < 0")
        if len(set(seq_ids)) != len(seq_ids):
            raise ValueError("a sequence appears twice")
        for s in seq_ids:
            self.block_table[s]
        if self._pages_needed(seq_ids, n_new) > len(self.free_list):
            raise OutOfBlocks()
        cow = []
        for s in seq_ids:
            table = self.block_table[s]
            L = self.length[s]
            for pos in range(L, L + n_new):
                idx = pos // self.page_size
                if idx >= len(table):
                    pid = self.free_list.pop()
                    self.ref_count[pid] = 1
                    table.append(pid)
                pid = table[idx]
                if self.ref_count[pid] > 1:
                    new_pid = self.free_list.pop()
                    cow.append((pid, new_pid))
                    self.ref_count[pid] -= 1
                    self.ref_count[new_pid] = 1
                    table[idx] = new_pid
            self.length[s] = L + n_new
        return cow

    # -- rollback ------------------------------------------------------------
    def truncate(self, seq_id, new_len):
        L = self.length[seq_id]
        if new_len < 0 or new_len > L:
            raise ValueError("new_len outside [0, len]")
        table = self.block_table[seq_id]
        keep = self._pages_for(new_len)
        for pid in table[keep:]:
            self._release(pid)
        del table[keep:]
        self.length[seq_id] = new_len

    def commit_verify(self, seq_ids, n_new, num_accepted):
        if len(set(seq_ids)) != len(seq_ids):
            raise ValueError("a sequence appears twice")
        targets = []
        for s, n in zip(seq_ids, num_accepted, strict=True):
            if n < 0 or n > n_new - 1:
                raise ValueError("num_accepted outside [0, n_new - 1]")
            if self.length[s] < n_new:
                raise ValueError("sequence shorter than the n_new rows of the round")
            new_len = self.length[s] - n_new + n + 1
            targets.append((s, new_len))
        for s, new_len in targets:
            self.truncate(s, new_len)

    # -- views -----------------------------------------------------------------
    def table(self, seq_ids, max_blocks):
        """Block table rows (padded with -1) and lengths, as plain lists."""
        rows, lens = [], []
        for s in seq_ids:
            pages = self.block_table[s]
            if len(pages) > max_blocks:
                raise ValueError("sequence needs more than max_blocks pages")
            rows.append(list(pages) + [-1] * (max_blocks - len(pages)))
            lens.append(self.length[s])
        return rows, lens
