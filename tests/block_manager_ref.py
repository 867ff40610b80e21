"""Plain-Python reference model of the host block manager, written from the pages
("推理框架知识点": vLLM BlockSpaceManagerV1.can_allocate / _allocate_sequence /
append_slots, the cached allocator and its LRU evictor; mlqm.cn article:
copy-on-write; nano-vLLM article §5.2.1: chain-hashed prefix blocks that keep
their token ids).  Used only by the tests, as the model the C++ manager is
compared with.

Policy choices both sides share (the pages leave them open): free blocks are a
stack initialised with ids 0..n-1 (the highest id is handed out first, freed
blocks are reused first); a released hashed block enters the evictor with the
next value of a global release counter and the evictor returns the smallest
one; full blocks only are identified by their prefix (the key here is the
tuple of all token ids up to and including the block, which is what the chain
hash stands for); swapping visits sequences in the given order and each
sequence's distinct blocks in increasing id order.
"""
from __future__ import annotations

OK, LATER, NEVER = 0, 1, 2


class _Pool:
    def __init__(self, n):
        self.ref = [0] * n
        self.key = [None] * n          # prefix key of a cached (hashed) block
        self.stamp = [None] * n        # evictor entry: release counter value
        self.free = list(range(n))
        self.by_key = {}

    def num_free(self):
        return len(self.free) + sum(1 for s in self.stamp if s is not None)

    def take(self):
        if self.free:
            b = self.free.pop()
        else:
            cands = [i for i, s in enumerate(self.stamp) if s is not None]
            if not cands:
                return None
            b = min(cands, key=lambda i: self.stamp[i])
            self.stamp[b] = None
            del self.by_key[self.key[b]]
            self.key[b] = None
        self.ref[b] = 1
        return b

    def release(self, b, counter):
        if self.ref[b] <= 0:
            return
        self.ref[b] -= 1
        if self.ref[b] == 0:
            if self.key[b] is not None:
                self.stamp[b] = counter()
            else:
                self.free.append(b)


class RefBlockManager:
    def __init__(self, bs, ngpu, ncpu=0, watermark=0.0, window=0, caching=False):
        self.bs, self.caching = bs, caching
        self.wb = -(-window // bs) if window > 0 else 0
        self.watermark_blocks = int(watermark * ngpu)
        self.ngpu = ngpu
        self.gpu, self.cpu = _Pool(ngpu), _Pool(ncpu)
        self.seqs = {}                 # id -> dict(table, tokens, swapped)
        self._counter = 0

    def _tick(self):
        self._counter += 1
        return self._counter

    def can_allocate(self, n):
        need = -(-n // self.bs)
        if self.wb:
            need = min(need, self.wb)
        if self.ngpu - need < self.watermark_blocks:
            return NEVER
        if self.gpu.num_free() - need >= self.watermark_blocks:
            return OK
        return LATER

    def _alloc_logical(self, s, i):
        if self.wb and i >= self.wb:
            return s["table"][i % self.wb]
        if self.caching and (i + 1) * self.bs <= len(s["tokens"]):
            key = tuple(s["tokens"][:(i + 1) * self.bs])
            b = self.gpu.by_key.get(key)
            if b is not None:
                self.gpu.stamp[b] = None
                self.gpu.ref[b] += 1
                return b
            b = self.gpu.take()
            if b is not None:
                self.gpu.key[b] = key
                self.gpu.by_key[key] = b
            return b
        return self.gpu.take()

    def allocate(self, sid, tokens):
        assert sid not in self.seqs
        s = {"table": [], "tokens": list(tokens), "swapped": False}
        for i in range(-(-len(tokens) // self.bs)):
            b = self._alloc_logical(s, i)
            if b is None:
                for x in sorted(set(s["table"])):
                    self.gpu.release(x, self._tick)
                raise MemoryError
            s["table"].append(b)
        self.seqs[sid] = s

    def append_slot(self, sid, token):
        s = self.seqs[sid]
        n = len(s["tokens"]) + 1
        cow = None
        if len(s["table"]) < -(-n // self.bs):
            if self.wb and len(s["table"]) >= self.wb:
                s["table"].append(s["table"][len(s["table"]) % self.wb])
            else:
                b = self.gpu.take()
                if b is None:
                    raise MemoryError
                s["table"].append(b)
        else:
            last = s["table"][-1]
            if self.gpu.ref[last] > 1:
                b = self.gpu.take()
                if b is None:
                    raise MemoryError
                s["table"][-1] = b
                self.gpu.release(last, self._tick)
                cow = (last, b)
        s["tokens"].append(token)
        last = s["table"][-1]
        if self.caching and n % self.bs == 0 and self.gpu.key[last] is None and self.gpu.ref[last] == 1:
            key = tuple(s["tokens"][:n])
            if key not in self.gpu.by_key:
                self.gpu.key[last] = key
                self.gpu.by_key[key] = last
        return last * self.bs + (n - 1) % self.bs, cow

    def fork(self, parent, child):
        p = self.seqs[parent]
        self.seqs[child] = {"table": list(p["table"]), "tokens": list(p["tokens"]), "swapped": False}
        for b in set(p["table"]):
            self.gpu.ref[b] += 1

    def free(self, sid):
        s = self.seqs.pop(sid)
        pool = self.cpu if s["swapped"] else self.gpu
        for b in sorted(set(s["table"])):
            pool.release(b, self._tick)

    def block_table(self, sid):
        s = self.seqs[sid]
        return list(s["table"]), len(s["tokens"])

    def _swap(self, sids, out):
        src, dst = (self.gpu, self.cpu) if out else (self.cpu, self.gpu)
        mapping = {}
        for sid in sids:
            s = self.seqs[sid]
            for b in sorted(set(s["table"])):
                if b in mapping:
                    dst.ref[mapping[b]] += 1
                else:
                    mapping[b] = dst.take()
                src.release(b, self._tick)
            s["table"] = [mapping[b] for b in s["table"]]
            s["swapped"] = out
        return sorted(mapping.items())

    def can_append_slots(self, num_running):
        return num_running <= self.gpu.num_free()

    def _distinct(self, sids, swapped):
        need = set()
        for sid in sids:
            s = self.seqs[sid]
            assert s["swapped"] == swapped
            need.update(s["table"])
        return len(need)

    def can_swap_in(self, sids):
        need = self._distinct(sids, True)
        if self.ngpu - need < self.watermark_blocks:
            return NEVER
        if self.gpu.num_free() - need >= self.watermark_blocks:
            return OK
        return LATER

    def can_swap_out(self, sids):
        return self._distinct(sids, False) <= self.cpu.num_free()

    def swap_out(self, sids):
        return self._swap(sids, True)

    def swap_in(self, sids):
        return self._swap(sids, False)
