"""The tcgen05 kernel's planner (tile height and K split), on the CPU through
the library's host-only test hook: the plans measured fastest on a GB300
(152 SMs) for the Llama-2 prefill layers, and the rules every plan keeps."""
import itertools

import pytest

SMS = 152


@pytest.fixture(scope="module")
def w4():
    import int4_weight_only_repack_gb300 as w4
    try:
        w4.lib()
    except OSError as e:  # the library is built by __graft_entry__.build()
        pytest.skip(f"library not built: {e}")
    return w4


# (M, N, K) -> (rows per tile, tiles, split tiles, K slices). Each plan was
# measured on a GB300 (graph-timed calls) against the alternatives named beside
# it, and was the fastest of them.
MEASURED_PLANS = [
    # 7B down, M = 512: 256-row tiles, all 32 split 4 ways (54 us; 128-row
    # tiles split 2 ways took 70 us)
    ((512, 4096, 11008), (256, 32, 32, 4)),
    # 70B gate_up, M = 128: one wave of whole tiles, the last 72 split in two
    # (142 us; unsplit 175 us, every tile split in two 159 us)
    ((128, 57344, 8192), (128, 224, 72, 2)),
    # 70B qkv, M = 128: 40 tiles split 3 ways fill one wave (41 us; 2 / 4 ways
    # 54 / 60 us, unsplit 90 us)
    ((128, 10240, 8192), (128, 40, 40, 3)),
    # 7B qkv, M = 4096: 5 waves + 8 tiles, the 8 split 8 ways (304 us; unsplit 335 us)
    ((4096, 12288, 4096), (256, 768, 8, 8)),
    # 7B qkv, M = 2048: 2 waves + 80 tiles; none split (171 us; the 80 split
    # 3 ways, their partials priced as if L2 kept them, 182 us)
    ((2048, 12288, 4096), (256, 384, 0, 1)),
    # 13B down, M = 1024: 80 tiles split 3 ways (175 us; 128-row tiles 220 us)
    ((1024, 5120, 13824), (256, 80, 80, 3)),
]


@pytest.mark.parametrize("shape,plan", MEASURED_PLANS)
def test_measured_plans(w4, shape, plan):
    assert w4.w4_test_prefill_plan(*shape, SMS) == plan


def test_plan_rules(w4):
    Ms = (17, 64, 65, 128, 129, 300, 512, 1000, 2048, 4096)
    Ns = (32, 256, 4096, 10240, 22016, 57344)
    Ks = (64, 512, 4096, 11008, 28672)
    for M, N, K, sms in itertools.product(Ms, Ns, Ks, (SMS, 148, 8)):
        rows, tiles, split_tiles, slices = w4.w4_test_prefill_plan(M, N, K, sms)
        assert rows in (128, 256)
        if M <= 128:
            assert rows == 128  # 256-row tiles only when a second accumulator has rows
        assert tiles == -(-M // rows) * -(-N // 256)
        assert 1 <= slices <= max(1, K // 64 // 8)  # slices of at least 8 k-blocks
        if slices == 1:
            assert split_tiles == 0
        else:
            # every tile when they cannot fill the SMs, else the last wave's few
            assert split_tiles == (tiles if tiles < sms else tiles % sms)
            assert split_tiles > 0


def test_plan_rejects_bad_shapes(w4):
    for args in [(16, 256, 256, SMS), (64, 100, 256, SMS), (64, 256, 100, SMS),
                 (64, 256, 256, 0), (1 << 21, 256, 256, SMS)]:
        with pytest.raises(w4.W4Error):
            w4.w4_test_prefill_plan(*args)
