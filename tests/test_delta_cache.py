"""Delta cache (bit_delta_compressed_gb300.cache): residency, LRU weighted by
request rate, pinning and single in-flight loads.  Host logic, tested on CPU
with a fake clock; one GPU test measures loads onto the device."""
import pytest
import torch

from bit_delta_compressed_gb300.cache import DeltaCache


class Clock:
    def __init__(self):
        self.t = 1000.0

    def __call__(self):
        return self.t


def host_variant(nbytes_bits, seed):
    g = torch.Generator().manual_seed(seed)
    bits = torch.randint(-2 ** 31, 2 ** 31, (nbytes_bits // 4,), generator=g, dtype=torch.int64).to(torch.int32)
    return [torch.rand(4, generator=g)], [bits]


def make(capacity, clock, n=4, size=1024):
    c = DeltaCache(capacity, "cpu", half_life_s=60.0, tau_s=30.0, clock=clock)
    for i in range(n):
        a, b = host_variant(size, i)
        c.register("v%d" % i, a, b)
    return c


def test_load_and_hit():
    clk = Clock()
    c = make(10 ** 6, clk)
    r = c.acquire("v1")
    a, b = c.host["v1"]
    assert torch.equal(r.bits[0], b[0]) and torch.equal(r.alphas[0], a[0])
    c.release(r)
    r2 = c.acquire("v1")
    assert r2 is r and c.stats["v1"].loads == 1 and c.stats["v1"].hits == 1
    c.release(r2)
    assert c.used == c.size_of("v1")


def test_lru_eviction_by_recency():
    clk = Clock()
    c = make(3 * (1024 + 16), clk)            # room for three variants
    for name in ("v0", "v1", "v2"):
        c.release(c.acquire(name))
        clk.t += 10
    c.release(c.acquire("v0"))                # v1 is now the least recently used
    clk.t += 10
    c.release(c.acquire("v3"))
    assert c.resident_names() == ["v0", "v2", "v3"]


def test_rate_weighting_keeps_hot_variant():
    clk = Clock()
    c = make(3 * (1024 + 16), clk)
    for _ in range(20):                       # v0 requested often, a while ago
        c.release(c.acquire("v0"))
        clk.t += 0.5
    clk.t += 20
    c.release(c.acquire("v1"))
    clk.t += 5
    c.release(c.acquire("v2"))
    clk.t += 5
    # v0: rate ~20, age 30 s; v1: rate 1, age 10 s -> v1 scores lower
    assert c.score("v0") > c.score("v1")
    c.release(c.acquire("v3"))
    assert "v0" in c.resident_names() and "v1" not in c.resident_names()


def test_pinned_variants_are_not_evicted():
    clk = Clock()
    c = make(2 * (1024 + 16), clk)
    r0 = c.acquire("v0")
    clk.t += 1
    r1 = c.acquire("v1")
    clk.t += 1
    with pytest.raises(MemoryError):
        c.acquire("v2")                        # both resident variants are in use
    c.release(r0)
    r2 = c.acquire("v2")                      # now v0 can go
    assert c.resident_names() == ["v1", "v2"]
    c.release(r1)
    c.release(r2)
    with pytest.raises(RuntimeError):
        c.release(r2)


def test_too_large_and_unknown():
    clk = Clock()
    c = make(100, clk)
    with pytest.raises(MemoryError):
        c.acquire("v0")
    with pytest.raises(KeyError):
        c.acquire("nope")


@pytest.mark.gpu
def test_gpu_loads_and_bandwidth():
    dev = torch.device("cuda", 0)
    nbits = 64 << 20                           # 64 MiB of bits per variant
    c = DeltaCache(3 * nbits + 4096, dev)
    hosts = {}
    for i in range(4):
        g = torch.Generator().manual_seed(i)
        bits = torch.randint(-2 ** 31, 2 ** 31, (nbits // 4,), generator=g, dtype=torch.int64).to(torch.int32)
        a = torch.rand(8, generator=g)
        hosts[i] = (a.pin_memory(), bits.pin_memory())
        c.register("v%d" % i, [hosts[i][0]], [hosts[i][1]])
    r = c.acquire("v0")
    torch.cuda.current_stream().synchronize()
    assert torch.equal(r.bits[0].cpu(), hosts[0][1]) and torch.equal(r.alphas[0].cpu(), hosts[0][0])
    c.release(r)
    # a load in flight is shared: the second acquire does not copy again
    r1 = c.acquire("v1")
    r1b = c.acquire("v1")
    assert r1b is r1 and c.stats["v1"].loads == 1
    c.release(r1)
    c.release(r1b)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(c.copy_stream)
    for name in ("v2", "v3"):
        c.release(c.acquire(name))
    t1.record(c.copy_stream)
    torch.cuda.synchronize()
    gbs = 2 * (nbits + 32) / (t0.elapsed_time(t1) / 1e3) / 1e9
    assert gbs > 1.0
    assert len(c.resident_names()) == 3
