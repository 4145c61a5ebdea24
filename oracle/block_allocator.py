"""Plain-Python model of the host block allocator -- TEST INFRASTRUCTURE ONLY.

The reference the library's allocator (pkv_allocator_*) is compared against,
operation by operation.  It follows "Paged KV Cache - AI infra interview
lesson" (Walk the Shapes First: slot = block_table[p // bs] * bs + p % bs and a
new block exactly when a position p has p % bs == 0; Append slots during
decode; Separate allocation, sharing and release: a block returns to the free
pool only after its final reference is released) and the accounting
invariants of "Chapter 2 -- KV cache, memory hierarchy, continuous batching,
and PagedAttention", Deterministic evals for this layer.  Free blocks are
handed out lowest-numbered first; a shared prefix is whole blocks.
"""
from __future__ import annotations


class AllocatorError(Exception):
    pass


class OutOfBlocks(AllocatorError):
    pass


class ModelAllocator:
    def __init__(self, num_blocks: int, block_size: int):
        self.num_blocks, self.bs = num_blocks, block_size
        self.ref = [0] * num_blocks
        self.seqs = {}  # id -> {"blocks": [...], "len": n}

    def _free(self):
        return [b for b in range(self.num_blocks) if self.ref[b] == 0]

    def _take(self, n):
        free = self._free()
        if n > len(free):
            raise OutOfBlocks(n)
        for b in free[:n]:
            self.ref[b] = 1
        return free[:n]

    def add_sequence(self, seq, num_tokens, blocks=None):
        if seq in self.seqs or num_tokens < 0:
            raise AllocatorError(seq)
        n = -(-num_tokens // self.bs)
        if blocks is not None:
            blocks = list(blocks)[:n]
            if len(set(blocks)) != n or any(not 0 <= b < self.num_blocks or self.ref[b] for b in blocks):
                raise AllocatorError(blocks)
            for b in blocks:
                self.ref[b] = 1
        else:
            blocks = self._take(n)
        self.seqs[seq] = {"blocks": blocks, "len": num_tokens}

    def fork(self, parent, child, num_tokens):
        if parent not in self.seqs or child in self.seqs:
            raise AllocatorError((parent, child))
        p = self.seqs[parent]
        if num_tokens < 0 or num_tokens > p["len"] or num_tokens % self.bs:
            raise AllocatorError(num_tokens)
        shared = p["blocks"][:num_tokens // self.bs]
        for b in shared:
            self.ref[b] += 1
        self.seqs[child] = {"blocks": list(shared), "len": num_tokens}

    def append(self, seq, num_tokens=1):
        s = self.seqs[seq] if seq in self.seqs else None
        if s is None or num_tokens < 0:
            raise AllocatorError(seq)
        need = -(-(s["len"] + num_tokens) // self.bs) - len(s["blocks"])
        if need > 0:
            s["blocks"] += self._take(need)
        slots = []
        for i in range(num_tokens):
            p = s["len"] + i
            slots.append(s["blocks"][p // self.bs] * self.bs + p % self.bs)
        s["len"] += num_tokens
        return slots

    def release(self, seq):
        if seq not in self.seqs:
            raise AllocatorError(seq)
        for b in self.seqs.pop(seq)["blocks"]:
            self.ref[b] -= 1

    def block_table(self, seq, max_blocks):
        s = self.seqs[seq]
        return s["blocks"] + [-1] * (max_blocks - len(s["blocks"])), s["len"], len(s["blocks"])

    def stats(self):
        referenced = {b for s in self.seqs.values() for b in s["blocks"]}
        allocated = sum(1 for r in self.ref if r > 0)
        return {"free": self.num_blocks - allocated, "allocated": allocated, "referenced": len(referenced),
                "sequences": len(self.seqs)}

    def check(self):
        """The page's accounting, restated: 0 when it holds, else the first
        broken rule (numbered as pkv_allocator_check numbers them)."""
        counts = [0] * self.num_blocks
        for s in self.seqs.values():
            if len(s["blocks"]) != -(-s["len"] // self.bs):
                return 5
            for b in s["blocks"]:
                counts[b] += 1
        if counts != self.ref:
            return 2
        st = self.stats()
        if st["free"] + st["allocated"] != self.num_blocks:
            return 1
        if st["allocated"] < st["referenced"]:
            return 3
        for s in self.seqs.values():
            if s["len"] % self.bs and counts[s["blocks"][-1]] != 1:
                return 4
        return 0
