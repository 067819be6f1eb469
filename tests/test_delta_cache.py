"""Delta cache (bit_delta_compressed_gb300.cache): residency, the hot set of
the most requested variants, LRU weighted by request rate for the rest,
pinning and single in-flight loads.  Host logic, tested on CPU with a fake
clock; the GPU tests check device contents through eviction and reload and
that evicted memory is reused only after the consuming stream's work."""
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


def make(capacity, clock, n=4, size=1024, top_k=0):
    # top_k = 0: the LRU tier alone (no hot set)
    c = DeltaCache(capacity, "cpu", half_life_s=60.0, tau_s=30.0, clock=clock, pinned_top_k=top_k)
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


SIZE = 1024 + 16                              # bytes of one test variant (bits + 4 scales)


def test_hot_set_survives_cold_pressure():
    # 14 variants, room for 7: the six most requested stay resident while the
    # eight others take turns in the one slot left (the page's 6 + 8 split)
    clk = Clock()
    c = make(7 * SIZE, clk, n=14, top_k=6)
    for rnd in range(10):
        for i in range(6):
            c.release(c.acquire("v%d" % i))
            clk.t += 0.1
    assert c.hot_set() == {"v%d" % i for i in range(6)}
    for i in range(6, 14):                    # eight cold variants, once each
        clk.t += 1.0
        c.release(c.acquire("v%d" % i))
        names = c.resident_names()
        assert all("v%d" % h in names for h in range(6)), names
        assert "v%d" % i in names and len(names) == 7
    # the cold tier alone evicted: every cold variant was loaded once
    assert all(c.stats["v%d" % i].loads == 1 for i in range(14))


def test_hot_variant_demoted_after_its_rate_decays():
    clk = Clock()
    c = make(3 * SIZE, clk, n=5, top_k=1)
    for _ in range(30):                       # v0 hot
        c.release(c.acquire("v0"))
        clk.t += 0.1
    for name in ("v1", "v2"):
        c.release(c.acquire(name))
    assert c.hot_set() == {"v0"}
    clk.t += 1.0
    c.release(c.acquire("v3"))                # evicts a cold one, never v0
    assert "v0" in c.resident_names()
    # ten half-lives later v0's rate has decayed below v4's fresh traffic
    clk.t += 600.0
    for _ in range(3):
        c.release(c.acquire("v4"))
        clk.t += 0.1
    assert c.hot_set() == {"v4"}
    for name in ("v1", "v2"):                 # pressure: v0 is now an ordinary variant
        clk.t += 1.0
        c.release(c.acquire(name))
    assert "v0" not in c.resident_names() and "v4" in c.resident_names()


def test_hot_set_ranks_by_rate_and_warm_loads_it():
    clk = Clock()
    c = make(4 * SIZE, clk, n=6, top_k=2)
    for name, reps in (("v0", 2), ("v1", 5), ("v2", 9), ("v3", 5)):
        for _ in range(reps):
            c.release(c.acquire(name))
    assert c.hot_set() == {"v2", "v1"}        # v1 and v3 tie on rate: name order
    c2 = make(4 * SIZE, clk, n=6, top_k=2)
    c2.stats = c.stats                        # same traffic, nothing resident yet
    assert c2.warm() == ["v2", "v1"] and c2.resident_names() == ["v1", "v2"]
    assert c2.warm() == []


def test_hot_set_cannot_be_evicted():
    clk = Clock()
    c = make(2 * SIZE, clk, n=3, top_k=2)
    for name in ("v0", "v1"):
        for _ in range(3):
            c.release(c.acquire(name))
    with pytest.raises(MemoryError):
        c.acquire("v2")                        # both residents are hot
    with pytest.raises(ValueError):
        DeltaCache(10, "cpu", pinned_top_k=-1)


def _gpu_variants(c, n, nbits):
    hosts = {}
    for i in range(n):
        g = torch.Generator().manual_seed(i)
        bits = torch.randint(-2 ** 31, 2 ** 31, (nbits // 4,), generator=g, dtype=torch.int64).to(torch.int32)
        a = torch.rand(8, generator=g)
        hosts[i] = (a.pin_memory(), bits.pin_memory())
        c.register("v%d" % i, [hosts[i][0]], [hosts[i][1]])
    return hosts


@pytest.mark.gpu
def test_gpu_contents_through_eviction_and_reload():
    dev = torch.device("cuda", 0)
    nbits = 16 << 20
    c = DeltaCache(2 * (nbits + 32) + 64, dev, pinned_top_k=0)
    hosts = _gpu_variants(c, 3, nbits)
    for cycle in range(2):                    # v0, v1 resident; v2 evicts one; reload it
        for i in (0, 1, 2, 0, 2, 1):
            r = c.acquire("v%d" % i)
            got_bits = r.bits[0].cpu()        # on the current stream, after the load
            got_a = r.alphas[0].cpu()
            assert torch.equal(got_bits, hosts[i][1]) and torch.equal(got_a, hosts[i][0]), (cycle, i)
            c.release(r)
            assert len(c.resident_names()) <= 2
    assert sum(c.stats["v%d" % i].loads for i in range(3)) > 3   # evictions happened


@pytest.mark.gpu
def test_gpu_evicted_memory_waits_for_the_consumer():
    # a consumer stream reads variant v0 behind a long sleep; v0 is then
    # evicted and v1 loaded into the freed space.  The consumer must still
    # read v0's bits: the freed block is reused only after its queued work.
    dev = torch.device("cuda", 0)
    nbits = 32 << 20
    c = DeltaCache(nbits + 32 + 64, dev, pinned_top_k=0)
    hosts = _gpu_variants(c, 2, nbits)
    consumer = torch.cuda.Stream(device=dev)
    r0 = c.acquire("v0", stream=consumer)
    with torch.cuda.stream(consumer):
        torch.cuda._sleep(200_000_000)        # ~0.1 s of GPU time before the read
        out = r0.bits[0].clone()
    c.release(r0)
    del r0
    r1 = c.acquire("v1")                      # evicts v0 while the consumer still waits
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), hosts[0][1])
    assert torch.equal(r1.bits[0].cpu(), hosts[1][1])
    c.release(r1)


@pytest.mark.gpu
def test_gpu_loads_and_bandwidth():
    dev = torch.device("cuda", 0)
    nbits = 64 << 20                           # 64 MiB of bits per variant
    c = DeltaCache(3 * nbits + 4096, dev, pinned_top_k=0)
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
