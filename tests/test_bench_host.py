"""Host-side pieces of bench.py (no GPU): the per-step spread and the kernel
source hashes that key the recorded ncu traffic."""

import bench


def test_spread_nearest_rank():
    xs = list(range(1, 101))            # 1..100
    sp = bench.spread(reversed(xs))
    assert sp == {"p10": 10.0, "median": 50.5, "p90": 90.0}
    assert bench.spread([7.0]) == {"p10": 7.0, "median": 7.0, "p90": 7.0}
    assert bench.spread([]) is None
    sp = bench.spread([3.0, 1.0, 2.0])
    assert sp["p10"] == 1.0 and sp["median"] == 2.0 and sp["p90"] == 3.0


def test_kernel_hashes_ignore_comments_and_key_the_traffic():
    for k in ("build", "verify", "attn"):
        h = bench._kernel_source_hash(k)
        assert len(h) == 12 and int(h, 16) >= 0
    # every recorded traffic figure belongs to a known kernel and workload
    for key, (h, nbytes) in bench.TRAFFIC.items():
        kernel, wl = key.split(":")
        assert kernel in bench.KERNEL_SOURCES and wl.startswith("c") and nbytes > 0
