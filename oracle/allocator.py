"""Free-block pool allocator, restated as plain Python lists.

Test infrastructure only (see the package docstring).

Semantics follow the paged KV-cache manager of [D] "连续批处理与KV缓存" §4.2:

* the pool starts as the list of all block ids, in order (or in a given
  order, which stands in for a pool that has already been shuffled by use);
* ``alloc(req, n)`` takes the first ``n`` ids off the front of the free list,
  all or nothing -- if fewer than ``n`` are free it fails ("OOM: wait or
  evict") and nothing changes;
* ``append_block(req)`` takes one id off the front, or reports that the pool
  is empty ("needs to wait");
* ``free(req)`` returns all of a request's blocks to the back of the free
  list, in the order the request held them.

Readings where the page is silent or its sketch is unsafe (each is listed in
the design notes):

* allocating an id that is already live is rejected (the page's dict
  assignment would silently overwrite the old list and leak its blocks);
* freeing or appending to an unknown id is rejected with no state change (the
  page's ``pop(req, [])`` ignores it; its ``append`` would raise);
* blocks shared by many requests (a common prompt prefix, [B] §3.2, [E] §2.1)
  are attached in front of a request's private blocks and are never returned
  by ``free`` -- whoever allocated them owns them.

Copy-on-write forking ([B] §3.2: requests with a common prefix point at the
same physical blocks, and a block is copied only when one of them must write
into it -- parallel sampling, beam search):

* ``fork(parent, child)`` gives the child the parent's whole table; every
  block the parent holds is now held by both. A block's reference count is
  the number of live requests whose own list holds it;
* ``cow(req, i)`` is called before a request writes into its logical block i:
  if that block is held by others too, the request takes a fresh block from
  the front of the free list in its place (the caller copies the contents
  over) and ``(old, new)`` is returned; a block held by the request alone
  needs no copy (``None``). Attached prefix blocks are read-only;
* ``free(req)`` drops the request's references and returns, in its order,
  only the blocks nobody holds any more.
"""

from __future__ import annotations


class OutOfBlocks(Exception):
    """Fewer free blocks than requested; the pool is unchanged."""


class UnknownRequest(KeyError):
    """The request id has no live allocation."""


class DuplicateRequest(KeyError):
    """The request id already has a live allocation."""


class FreeBlockPool:
    def __init__(self, total_blocks: int, initial_order=None):
        if initial_order is None:
            initial_order = range(total_blocks)
        order = [int(b) for b in initial_order]
        if sorted(order) != list(range(total_blocks)):
            raise ValueError("initial_order must be a permutation of range(total_blocks)")
        self.total_blocks = total_blocks
        self.free_list = order          # front = next block handed out
        self.private = {}               # req -> [block ids it owns, in order]
        self.shared = {}                # req -> [pinned block ids it references]

    # -- the three operations of the page ---------------------------------
    def alloc(self, req: int, n: int) -> list:
        if n < 0:
            raise ValueError("n must be >= 0")
        if req in self.private:
            raise DuplicateRequest(req)
        if len(self.free_list) < n:
            raise OutOfBlocks(req)
        taken = self.free_list[:n]
        self.free_list = self.free_list[n:]
        self.private[req] = list(taken)
        self.shared[req] = []
        return list(taken)

    def free(self, req: int) -> list:
        if req not in self.private:
            raise UnknownRequest(req)
        held = self.private.pop(req)
        self.shared.pop(req)
        returned = [b for b in held if self.refs(b) == 0]
        self.free_list.extend(returned)
        return returned

    def append_block(self, req: int):
        """Returns the new block id, or None when the pool is empty."""
        if req not in self.private:
            raise UnknownRequest(req)
        if not self.free_list:
            return None
        block = self.free_list.pop(0)
        self.private[req].append(block)
        return block

    # -- shared prefix blocks ---------------------------------------------
    def attach_shared(self, req: int, ids) -> None:
        if req not in self.private:
            raise UnknownRequest(req)
        self.shared[req] = [int(b) for b in ids] + self.shared[req]

    # -- copy-on-write forking ---------------------------------------------
    def refs(self, block: int) -> int:
        """Live requests whose own block list holds ``block``."""
        return sum(block in held for held in self.private.values())

    def fork(self, parent: int, child: int) -> None:
        if parent not in self.private:
            raise UnknownRequest(parent)
        if child in self.private:
            raise DuplicateRequest(child)
        self.private[child] = list(self.private[parent])
        self.shared[child] = list(self.shared[parent])

    def cow(self, req: int, index: int):
        """Before ``req`` writes into its logical block ``index``: None if the
        block is its alone, else (old, new) after swapping in a fresh block."""
        if req not in self.private:
            raise UnknownRequest(req)
        k = index - len(self.shared[req])
        if k < 0:
            raise ValueError("attached prefix blocks are read-only")
        old = self.private[req][k]
        if self.refs(old) <= 1:
            return None
        if not self.free_list:
            raise OutOfBlocks(req)
        new = self.free_list.pop(0)
        self.private[req][k] = new
        return old, new

    # -- views -------------------------------------------------------------
    def table(self, req: int) -> list:
        """Logical block i of the request -> physical block id."""
        if req not in self.private:
            raise UnknownRequest(req)
        return self.shared[req] + self.private[req]

    def num_free(self) -> int:
        return len(self.free_list)

    def block_tables(self, reqs, max_blocks: int):
        """Rows of physical ids, padded with -1 to ``max_blocks`` columns."""
        rows = []
        for r in reqs:
            t = self.table(r)
            if len(t) > max_blocks:
                raise ValueError("request holds more blocks than max_blocks")
            rows.append(t + [-1] * (max_blocks - len(t)))
        return rows
