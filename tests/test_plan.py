"""The plan chooser's decisions, without a device (gemm_plan_query with a
GB300's 152 SMs, 76 co-resident CTA pairs and 36 clusters of two pairs).

Each case pins a choice that measurements on GB300 showed to be the fastest
(or within 2% of it) among the kernel families and tile widths, so that a
change of the cost tables that moves it fails here before it reaches a GPU.
"""

import pytest

from dense_gemm_tensor_gb300 import build, gemm

SINGLE, PAIR, PAIR_ON_CT, TWO_PAIRS = 1, 2, 3, 4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    gemm.load()
    gemm.set_tuning(0, 0, 0, 0)
    yield
    gemm.set_tuning(0, 0, 0, 0)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "tf32"])
def test_4096_row_major_b_takes_the_transposed_product(dtype):
    """4096^3, row-major B: the pair on C^T with 224-row tiles (seven stages),
    four whole rounds, bands of 16 tile rows (BF16 82.6 against 84.4 us for
    the plain pair; TF32 154.9 against 157.2)."""
    p = gemm.plan_query(dtype, 4096, 4096, 4096)
    assert (p["kernel"], p["tile_n"], p["raster"], p["tail_segs"]) == (PAIR_ON_CT, 224, 16, 1)
    assert p["grid"] == 152 and p["concurrent_tiles"] == 76


@pytest.mark.parametrize("dtype", ["bf16", "tf32"])
def test_4096_k_major_b_takes_the_plain_pair(dtype):
    """K-major B has no unused box columns: the plain pair, 224 wide."""
    p = gemm.plan_query(dtype, 4096, 4096, 4096, layout=gemm.GEMM_B_K_MAJOR)
    assert (p["kernel"], p["tile_n"], p["tail_segs"]) == (PAIR, 224, 1)


def test_fused_call_keeps_the_plain_pair():
    """A fused epilogue is costlier on the transposed product (beta * C:
    100.2 against 97.4 us): fused calls stay on the plain pair."""
    p = gemm.plan_query("bf16", 4096, 4096, 4096, fused=True)
    assert (p["kernel"], p["tile_n"]) == (PAIR, 224)


def test_8192_splits_the_last_round():
    """8192^3: 256-wide pair tiles, 1024 tiles = 13 rounds + 36, the last
    round split in two along K."""
    p = gemm.plan_query("bf16", 8192, 8192, 8192)
    assert (p["kernel"], p["tile_n"], p["tail_segs"]) == (PAIR, 256, 2)


def test_projection_and_fp8():
    p = gemm.plan_query("bf16", 8192, 28672, 8192, layout=gemm.GEMM_B_K_MAJOR)
    assert (p["kernel"], p["tile_n"], p["tail_segs"]) == (PAIR, 256, 4)
    p = gemm.plan_query("e4m3", 8192, 8192, 8192, layout=gemm.GEMM_B_K_MAJOR)
    assert (p["kernel"], p["tile_n"], p["tail_segs"]) == (PAIR, 256, 2)


def test_ragged_row_major_b_keeps_the_plain_pair():
    """4000 x 4100 x 4104: 4100 columns would leave a 256-column block of C
    nearly empty on the transposed product; the plain 224-wide pair fills four
    rounds exactly."""
    p = gemm.plan_query("bf16", 4000, 4100, 4104)
    assert (p["kernel"], p["tile_n"]) == (PAIR, 224)


def test_small_products_and_batches_take_the_single_cta_kernel():
    # narrow tiles spread a small product over more SMs (CUDA graphs on GB300:
    # 512^3 5.23 us at 32 wide against 6.17 at 128; 1024^3 8.00 at 64 against
    # 8.62 at 128 and 12.26 at 32)
    p = gemm.plan_query("bf16", 512, 512, 512)
    assert (p["kernel"], p["tile_n"]) == (SINGLE, 32)
    p = gemm.plan_query("bf16", 1024, 1024, 1024)
    assert (p["kernel"], p["tile_n"]) == (SINGLE, 64)
    assert gemm.plan_query("bf16", 2048, 2048, 2048)["kernel"] == SINGLE  # 21.2 against 23.2 us
    p = gemm.plan_query("bf16", 512, 512, 512, batch=128)  # 45.8 us against 53.9 on the pair
    assert (p["kernel"], p["tile_n"]) == (SINGLE, 256)


def test_tf32_2048_row_major_b_avoids_the_single_cta_kernel():
    """TF32 with row-major B fetches B in 32-column boxes: at 2048^3 the
    single-CTA kernel ran 38.6 us, a pair plan 33.4-34.0."""
    assert gemm.plan_query("tf32", 2048, 2048, 2048)["kernel"] in (PAIR, TWO_PAIRS)


def test_two_pairs_only_where_their_clusters_fit_whole_rounds():
    """Clusters of two pairs cost about 1.2 us more per launch than single
    pairs with the same rounds (BF16 3072^3: 35.2 against 34.1 us on GB300;
    2048 x 2048 x 8192: 44.5 against 43.2); at 6144^3 with K-major B their 36
    clusters fill eight whole rounds and they were faster (242.8 against
    250.3 us)."""
    assert gemm.plan_query("bf16", 3072, 3072, 3072)["kernel"] == PAIR
    assert gemm.plan_query("bf16", 2048, 2048, 8192)["kernel"] == PAIR
    assert gemm.plan_query("tf32", 2048, 2048, 2048)["kernel"] == PAIR
    assert gemm.plan_query("bf16", 6144, 6144, 6144, layout=gemm.GEMM_B_K_MAJOR)["kernel"] == TWO_PAIRS


def test_short_tails_stay_unsplit():
    """Splitting the last round costs about 4 us per segment (partials out
    and back): TF32 2560^3 ran 55.6 us split in three against 48.8 unsplit on
    192-wide tiles; BF16 12288 x 4096 x 4096 with K-major B 237.5 split in
    four against 221.3 unsplit on 224-wide tiles."""
    p = gemm.plan_query("tf32", 2560, 2560, 2560)
    assert (p["kernel"], p["tile_n"], p["tail_segs"]) == (PAIR_ON_CT, 192, 1)
    p = gemm.plan_query("bf16", 12288, 4096, 4096, layout=gemm.GEMM_B_K_MAJOR)
    assert (p["kernel"], p["tile_n"], p["tail_segs"]) == (PAIR, 224, 1)


def test_tuning_hook_forces_the_plan():
    gemm.set_tuning(4, 256, 0, 0)
    try:
        p = gemm.plan_query("bf16", 4096, 4096, 4096)
        assert (p["kernel"], p["tile_n"]) == (PAIR_ON_CT, 256)
        # the transposed product exists for row-major B only: forcing it for
        # K-major B falls back to the single-CTA default
        assert gemm.plan_query("bf16", 4096, 4096, 4096, layout=gemm.GEMM_B_K_MAJOR)["kernel"] == SINGLE
    finally:
        gemm.set_tuning(0, 0, 0, 0)


def test_plan_query_rejects_bad_arguments():
    import ctypes
    lib = gemm.load()
    out = (ctypes.c_int32 * 6)()
    assert lib.gemm_plan_query(7, 64, 64, 64, 0, 1, 0, 152, 76, 36, out) == gemm.GEMM_ERR_INVALID_VALUE
    assert lib.gemm_plan_query(1, 0, 64, 64, 0, 1, 0, 152, 76, 36, out) == gemm.GEMM_ERR_INVALID_VALUE
    assert lib.gemm_plan_query(1, 64, 64, 64, 2, 1, 0, 152, 76, 36, out) == gemm.GEMM_ERR_INVALID_VALUE
    assert lib.gemm_plan_query(1, 64, 64, 64, 0, 1, 0, 152, 0, 36, out) == gemm.GEMM_ERR_INVALID_VALUE
    assert lib.gemm_plan_query(1, 64, 64, 64, 0, 1, 0, 152, 76, 36, None) == gemm.GEMM_ERR_INVALID_VALUE
