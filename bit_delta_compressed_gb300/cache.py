"""Device residency of variant deltas (the delta cache).

Page: "BitDelta: serving 14 Zen models from one GPU cluster", section
"Infrastructure details": each variant's deltas (packed sign bits and f32
scales) live in host storage and are loaded onto the GPU on first use; the
GPU keeps the variants in use, keeping the most requested ones resident at all
times and sharing the rest of the space among the others by recency and
request rate (the cache-eviction paragraph: the six variants with the most
traffic always stay loaded, the remaining eight share what is left under
LRU).

``DeltaCache`` holds the device copies within a byte budget:

* ``register(name, alphas, bits)``: a variant's host copies (pinned CPU
  tensors: one f32 scale tensor and one packed-bits tensor per matrix).
* ``acquire(name)``: makes the variant resident and returns a ``Resident``
  whose ``alphas`` / ``bits`` are device tensors; the caller's stream waits
  for the load (if one is in flight) before it uses them.  A variant being
  loaded is loaded once: concurrent acquires share the in-flight copy.
  Acquired variants are pinned (not evictable) until ``release``.
* The hot set: the ``pinned_top_k`` registered variants with the highest
  request rate (an exponentially decayed request count, ties broken by name)
  are never evicted.  The ranking is taken afresh at every eviction, so a
  variant whose traffic fades drops out of the hot set and becomes evictable,
  and one whose traffic grows joins it.  ``warm()`` loads every hot variant
  that is not resident.
* Eviction, when a load needs room: among resident variants that are neither
  hot nor acquired and whose copy has completed, the one with the smallest
  score = request rate x recency weight, recency exp(-age / tau); if only
  in-flight ones qualify, the oldest copy is waited for first.  When nothing
  qualifies the load raises MemoryError.

Copies run on a stream of their own (host-to-device from pinned memory), so a
load overlaps compute on the caller's stream; the device tensors are marked as
used on the caller's stream, so memory freed by an eviction is reused only
after the work queued there has finished.  On a CPU "device" the same logic
runs with plain copies (used by the host-side tests).
"""
from __future__ import annotations

import math
import time
from dataclasses import dataclass


@dataclass
class Resident:
    name: str
    alphas: list
    bits: list
    nbytes: int
    ready: object = None            # torch.cuda.Event (None on a host-only device)
    pins: int = 0
    loading: bool = False


@dataclass
class _Stats:
    rate: float = 0.0
    last: float = 0.0
    hits: int = 0
    loads: int = 0


class DeltaCache:
    def __init__(self, capacity_bytes: int, device, half_life_s: float = 60.0, tau_s: float = 30.0,
                 clock=time.monotonic, pinned_top_k: int = 6):
        import torch
        self.torch = torch
        self.capacity = int(capacity_bytes)
        self.device = torch.device(device)
        self.half_life = float(half_life_s)
        self.tau = float(tau_s)
        self.clock = clock
        if pinned_top_k < 0:
            raise ValueError("pinned_top_k must be >= 0")
        self.pinned_top_k = int(pinned_top_k)
        self.host: dict[str, tuple[list, list]] = {}
        self.resident: dict[str, Resident] = {}
        self.stats: dict[str, _Stats] = {}
        self.used = 0
        self.bytes_loaded = 0
        self.cuda = self.device.type == "cuda"
        self.copy_stream = torch.cuda.Stream(device=self.device) if self.cuda else None

    # -- registration -------------------------------------------------------------
    def register(self, name: str, alphas: list, bits: list) -> None:
        if len(alphas) != len(bits):
            raise ValueError("one scale tensor per bits tensor")
        for t in list(alphas) + list(bits):
            if t.device.type != "cpu":
                raise ValueError("host copies must be CPU tensors")
        self.host[name] = (list(alphas), list(bits))
        self.stats.setdefault(name, _Stats())

    @staticmethod
    def _nbytes(tensors) -> int:
        return sum(t.numel() * t.element_size() for t in tensors)

    def size_of(self, name: str) -> int:
        a, b = self.host[name]
        return self._nbytes(a) + self._nbytes(b)

    # -- scoring --------------------------------------------------------------------
    def _touch(self, name: str, now: float) -> None:
        st = self.stats[name]
        if st.last > 0.0:
            st.rate *= math.pow(0.5, max(0.0, now - st.last) / self.half_life)
        st.rate += 1.0
        st.last = now

    def rate(self, name: str, now: float | None = None) -> float:
        """Request rate: the decayed request count, decayed to ``now``."""
        now = self.clock() if now is None else now
        st = self.stats[name]
        return st.rate * math.pow(0.5, max(0.0, now - st.last) / self.half_life)

    def score(self, name: str, now: float | None = None) -> float:
        """Request rate (decayed to ``now``) times the recency weight."""
        now = self.clock() if now is None else now
        age = max(0.0, now - self.stats[name].last)
        return self.rate(name, now) * math.exp(-age / self.tau)

    def hot_set(self, now: float | None = None) -> set:
        """The ``pinned_top_k`` registered variants with the highest request
        rate (variants never requested are not ranked)."""
        now = self.clock() if now is None else now
        ranked = sorted((n for n in self.stats if self.stats[n].rate > 0.0),
                        key=lambda n: (-self.rate(n, now), n))
        return set(ranked[:self.pinned_top_k])

    def _evict_for(self, need: int, now: float) -> None:
        self.poll()
        hot = self.hot_set(now)
        while self.used + need > self.capacity:
            free = [r for r in self.resident.values() if r.pins == 0 and r.name not in hot]
            cands = [r for r in free if not r.loading]
            if not cands:
                # variants whose copies are still in flight become evictable
                # once their copy completes: wait for the oldest
                waiting = [r for r in free if r.loading]
                if not waiting:
                    raise MemoryError("delta cache: %d bytes needed, %d free and nothing evictable "
                                      "(hot set %s)" % (need, self.capacity - self.used, sorted(hot)))
                waiting[0].ready.synchronize()
                self.poll()
                continue
            victim = min(cands, key=lambda r: (self.score(r.name, now), r.name))
            self._drop(victim)

    def _drop(self, r: Resident) -> None:
        del self.resident[r.name]
        self.used -= r.nbytes

    # -- acquire / release ------------------------------------------------------------
    def acquire(self, name: str, stream=None) -> Resident:
        """Resident copies of ``name``; ``stream`` (default: the current
        stream) waits for an in-flight load before its next work."""
        if name not in self.host:
            raise KeyError(name)
        now = self.clock()
        self._touch(name, now)
        r = self.resident.get(name)
        if r is None:
            r = self._load(name, now)
        else:
            self.stats[name].hits += 1
        r.pins += 1
        if self.cuda:
            s = stream if stream is not None else self.torch.cuda.current_stream(self.device)
            if r.ready is not None:
                s.wait_event(r.ready)
            # the allocator reuses the memory of an evicted variant only after
            # the work queued on ``s`` so far is done
            for t in r.alphas + r.bits:
                t.record_stream(s)
        return r

    def release(self, r: Resident) -> None:
        if r.pins <= 0:
            raise RuntimeError("release without acquire: " + r.name)
        r.pins -= 1

    def _load(self, name: str, now: float) -> Resident:
        torch = self.torch
        ha, hb = self.host[name]
        need = self.size_of(name)
        if need > self.capacity:
            raise MemoryError("variant %s (%d bytes) exceeds the cache (%d bytes)" % (name, need, self.capacity))
        self._evict_for(need, now)
        r = Resident(name=name, alphas=[], bits=[], nbytes=need, loading=True)
        self.resident[name] = r
        self.used += need
        if self.cuda:
            with torch.cuda.stream(self.copy_stream):
                r.alphas = [t.to(self.device, non_blocking=True) for t in ha]
                r.bits = [t.to(self.device, non_blocking=True) for t in hb]
                r.ready = torch.cuda.Event()
                r.ready.record(self.copy_stream)
        else:
            r.alphas = [t.clone() for t in ha]
            r.bits = [t.clone() for t in hb]
        if not self.cuda:
            r.loading = False
        self.stats[name].loads += 1
        self.bytes_loaded += need
        return r

    def warm(self) -> list:
        """Load every variant of the hot set that is not resident (without
        counting a request); returns the names loaded."""
        now = self.clock()
        loaded = []
        for name in sorted(self.hot_set(now), key=lambda n: (-self.rate(n, now), n)):
            if name not in self.resident:
                self._load(name, now)
                loaded.append(name)
        return loaded

    def poll(self) -> None:
        """Mark finished loads (their copies are complete) as evictable."""
        for r in self.resident.values():
            if r.loading and (r.ready is None or r.ready.query()):
                r.loading = False

    def resident_names(self) -> list:
        return sorted(self.resident)
