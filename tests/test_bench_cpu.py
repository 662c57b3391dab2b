"""The benchmark's own byte counts (its roofline bookkeeping, kept apart from the oracle)
equal the oracle's region split and step-bytes model."""

import itertools

import oracle

import bench


def test_regions_and_block_regions_match_the_oracle():
    for L, ns, nl in itertools.product([0, 1, 4, 5, 100, 131, 132, 133, 3000, 32768], [0, 4, 16], [0, 64, 128, 512]):
        assert bench.regions(L, ns, nl) == oracle.regions(L, ns, nl)
        assert bench.block_regions(L, ns, nl, 16) == oracle.block_regions(L, ns, nl, 16)


def test_step_bytes_match_the_oracle():
    for args in [(8, 8, 64, 128, 32768, 3277, 4, 128), (1, 8, 32, 128, 1048576, 100, 16, 512),
                 (2, 2, 16, 128, 100, 300, 4, 128), (1, 1, 8, 128, 4096, 256, 4, 64)]:
        assert bench.decode_step_hbm_bytes(*args) == oracle.decode_step_hbm_bytes(*args)
        assert (bench.decode_step_hbm_bytes(*args, per_query_head=True)
                == oracle.decode_step_hbm_bytes(*args, per_query_head=True))
