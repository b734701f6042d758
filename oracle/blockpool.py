"""The KV block allocator rule (test infrastructure).

ferrum-kernels ``cuda_decode.rs`` ``alloc_block``: a block is taken from the free list first
(last freed, first reused), otherwise the next never-used id is handed out; when neither is
possible the pool is exhausted and allocation fails. ``release_kv_cache`` returns a
sequence's blocks to the free list.
"""
from __future__ import annotations


class PoolExhausted(RuntimeError):
    pass


class BlockPool:
    def __init__(self, num_blocks: int):
        self.num_blocks = int(num_blocks)
        self.free = []            # a stack: the last block freed is the first reused
        self.next_id = 0

    def alloc(self) -> int:
        if self.free:
            return self.free.pop()
        if self.next_id < self.num_blocks:
            i = self.next_id
            self.next_id += 1
            return i
        raise PoolExhausted("KV block pool exhausted")

    def release(self, ids):
        for i in ids:
            self.free.append(int(i))

    def in_use(self) -> int:
        return self.next_id - len(self.free)
