"""Oracle model of the host page allocator.

TEST INFRASTRUCTURE ONLY: only the tests import it.  It shares nothing with
the library's allocator (csrc/alloc.cu); it restates the rules as literally
as possible, with plain lists and linear scans, so that a reader can check it
against them by eye:

  - tinyllm, "The repository currently provides": one runner-owned physical
    KV page pool, a worker-owned allocator and a logical block table per
    active sequence, with deterministic reserve/commit/release;
  - tinyllm, "Known limitations": 16-token pages; only complete pages are
    shared, a non-aligned suffix is recomputed;
  - Leone (introduction; "What ships"): page-rounded KV admission that
    returns typed overload errors before the configured capacity is
    exceeded; forked generation sessions.

Readings (the pages give no interface): a sequence holds
ceil((committed + reserved) / 16) pages; new pages are the lowest free ids,
appended in increasing order; an admission that cannot be met changes
nothing and raises CapacityError; fork shares the parent's complete committed
pages and nothing else; ids of sequences are the lowest closed ones.
"""
from __future__ import annotations

PAGE = 16


class CapacityError(Exception):
    """Typed overload: the pool (or a sequence's table) cannot take the pages."""


class ArgError(Exception):
    """A call the rules do not allow (unknown sequence, bad count)."""


def pages_for(tokens: int) -> int:
    return -(-tokens // PAGE)


class Allocator:
    def __init__(self, num_pages: int, max_seqs: int, max_pages_per_seq: int):
        if num_pages < 1 or max_seqs < 1 or max_pages_per_seq < 1:
            raise ArgError("sizes must be >= 1")
        self.num_pages, self.max_seqs, self.max_pages = num_pages, max_seqs, max_pages_per_seq
        self.refs = [0] * num_pages
        self.seqs: dict[int, dict] = {}  # open sequences: {"committed", "reserved", "pages"}

    # -- helpers, by definition --------------------------------------------
    def _free_ids(self):
        return [p for p in range(self.num_pages) if self.refs[p] == 0]

    def _seq(self, s):
        if s not in self.seqs:
            raise ArgError(f"sequence {s} is not open")
        return self.seqs[s]

    def _lowest_closed(self):
        for s in range(self.max_seqs):
            if s not in self.seqs:
                return s
        raise CapacityError("every sequence id is open")

    # -- the operations ------------------------------------------------------
    def open(self) -> int:
        s = self._lowest_closed()
        self.seqs[s] = {"committed": 0, "reserved": 0, "pages": []}
        return s

    def reserve(self, s: int, n: int):
        q = self._seq(s)
        if n < 0:
            raise ArgError("negative count")
        want = pages_for(q["committed"] + q["reserved"] + n)
        need = want - len(q["pages"])
        if want > self.max_pages:
            raise CapacityError("sequence would exceed max_pages_per_seq")
        free = self._free_ids()
        if need > len(free):
            raise CapacityError("not enough free pages")
        for p in free[:max(need, 0)]:
            self.refs[p] += 1
            q["pages"].append(p)
        q["reserved"] += n

    def commit(self, s: int, n: int):
        q = self._seq(s)
        if not 0 <= n <= q["reserved"]:
            raise ArgError("commit count outside [0, reserved]")
        q["committed"] += n
        q["reserved"] -= n

    def unreserve(self, s: int, n: int):
        q = self._seq(s)
        if not 0 <= n <= q["reserved"]:
            raise ArgError("unreserve count outside [0, reserved]")
        q["reserved"] -= n
        keep = pages_for(q["committed"] + q["reserved"])
        for p in q["pages"][keep:]:
            self.refs[p] -= 1
        del q["pages"][keep:]

    def fork(self, parent: int) -> int:
        p = self._seq(parent)
        full = p["committed"] // PAGE
        c = self._lowest_closed()
        shared = list(p["pages"][:full])
        for pg in shared:
            self.refs[pg] += 1
        self.seqs[c] = {"committed": full * PAGE, "reserved": 0, "pages": shared}
        return c

    def release(self, s: int):
        q = self._seq(s)
        for p in q["pages"]:
            self.refs[p] -= 1
        del self.seqs[s]

    def reserve_many(self, seqs, n: int):
        """Every sequence gets n more slots, or none does."""
        if n < 0 or len(set(seqs)) != len(seqs):
            raise ArgError("negative count or repeated sequence")
        for s in seqs:
            self._seq(s)
        import copy
        saved = copy.deepcopy((self.refs, self.seqs))
        try:
            for s in seqs:
                self.reserve(s, n)
        except (CapacityError, ArgError):
            self.refs, self.seqs = saved
            raise

    def commit_many(self, seqs, n: int):
        if n < 0 or len(set(seqs)) != len(seqs):
            raise ArgError("negative count or repeated sequence")
        for s in seqs:
            if n > self._seq(s)["reserved"]:
                raise ArgError("commit count above reserved")
        for s in seqs:
            self.commit(s, n)

    # -- views ------------------------------------------------------------------
    def info(self, s: int):
        q = self._seq(s)
        return q["committed"], q["reserved"], len(q["pages"])

    def block_table(self, s: int, stride: int):
        pages = self._seq(s)["pages"]
        if stride < len(pages):
            raise ArgError("stride below the page count")
        return pages + [-1] * (stride - len(pages))

    def batch(self, seqs, extra: int, stride: int):
        rows, lens = [], []
        for s in seqs:
            q = self._seq(s)
            if extra < 0 or extra > q["reserved"]:
                raise ArgError("extra outside [0, reserved]")
            rows.append(self.block_table(s, stride))
            lens.append(q["committed"] + extra)
        return rows, lens

    def stats(self):
        free = sum(1 for r in self.refs if r == 0)
        used = sum(1 for r in self.refs if r >= 1)
        shared = sum(1 for r in self.refs if r >= 2)
        return free, used, shared
