"""The split-over-keys plan (host logic, no GPU): which query blocks share
their keys among CTAs, checked through the C-ABI's fa_split_plan for a
152-SM GPU against the kernel's schedule and the cost it is meant to cut."""
import math

import pytest

import attention_forward_fwd_gb300 as fa

SMS = 152


def _block_tiles(qb, S, causal):
    """Key tiles (of 128) query block qb (256 rows) visits."""
    nkv = (S + 127) // 128
    n = 0
    for t in range(2):
        r0 = qb * 256 + t * 128
        if r0 < S:
            n = max(n, min(nkv, (r0 + 127) // 128 + 1) if causal else nkv)
    return n


@pytest.fixture(scope="module", autouse=True)
def built():
    fa.build()


@pytest.mark.parametrize("B,H,S,D,causal", [
    (4, 16, 4096, 64, True),      # 1024 blocks, many waves
    (2, 16, 8192, 128, True),
    (2, 16, 8192, 128, False),
    (1, 1, 256, 64, False),       # one key-tile pair: nothing to split
])
def test_full_shapes_are_not_split(B, H, S, D, causal):
    splits, items = fa.fa_split_plan(B, H, S, D, causal, SMS)
    assert set(splits) == {1}
    assert items == (S + 255) // 256


@pytest.mark.parametrize("causal", [False, True])
def test_one_head_splits_into_one_wave(causal):
    """B1 H1 S4096: 16 blocks on 152 SMs; the keys are split so that the
    items fill at most one wave, with chunks of at least two key tiles."""
    splits, items = fa.fa_split_plan(1, 1, 4096, 64, causal, SMS)
    assert max(splits) > 1 and items <= SMS
    assert items == sum(splits)
    for qb, n in enumerate(splits):
        assert 1 <= n <= _block_tiles(qb, 4096, causal)
        assert math.ceil(_block_tiles(qb, 4096, causal) / n) >= 2 or n == 1
    if not causal:
        assert splits == [8] * 16     # 32 key tiles in chunks of 4: 128 CTAs


@pytest.mark.parametrize("S", [1000, 4096])
@pytest.mark.parametrize("causal", [False, True])
def test_wide_kernel_splits_every_tile_alike(S, causal):
    """D > 128 (one CTA per 128-row query tile): B1 H2 leaves most SMs idle,
    so every tile's keys are divided into the same number of chunks (at most
    16, the merge kernel's register-held splits), filling at most one wave;
    a shape that fills the SMs is not split."""
    splits, items = fa.fa_split_plan(1, 2, S, 256, causal, SMS)
    ntq, max_kt = (S + 127) // 128, (S + 127) // 128
    ns = splits[0]
    assert 2 <= ns <= 16 and set(splits) == {ns}
    assert items == ntq * ns and 2 * items <= SMS
    chunk = math.ceil(max_kt / ns)
    assert math.ceil(max_kt / chunk) == ns      # no split past the last key tile
    full, items_full = fa.fa_split_plan(2, 16, 4096, 256, causal, SMS)
    assert set(full) == {1} and items_full == (4096 + 255) // 256


@pytest.mark.parametrize("causal", [False, True])
def test_wide_splits_fit_the_static_scratch(causal):
    """Every split plan of the wide kernel keeps at most one CTA per SM, so
    its partials (128 x 256 fp32 values plus m and l per CTA) fit the static
    entry point's 24 MiB scratch, whatever the shape."""
    worst = 0
    for B in (1, 2, 3):
        for H in (1, 2, 3, 5, 8):
            for S in (129, 256, 1000, 2048, 4096, 8192, 16384):
                splits, items = fa.fa_split_plan(B, H, S, 256, causal, SMS)
                if max(splits) == 1:
                    continue
                ctas = B * H * items
                assert ctas <= SMS
                worst = max(worst, ctas * (128 * 256 + 2 * 128) * 4)
    assert 0 < worst <= 24 << 20


def test_ragged_last_wave_is_split():
    """B3 H8 S1999 non-causal: 192 equal blocks on 152 SMs leave a second
    wave of 40; splitting some blocks shortens the schedule."""
    splits, items = fa.fa_split_plan(3, 8, 1999, 64, False, SMS)
    assert max(splits) > 1
    assert min(splits) == 1           # not every block pays for the merge
    assert items == sum(splits) <= 256


@pytest.mark.parametrize("B,H,S,D,causal", [
    (3, 8, 1999, 64, False), (3, 8, 1999, 64, True), (1, 1, 4096, 64, True),
    (1, 2, 3000, 64, True), (2, 3, 5000, 128, False), (1, 1, 300, 64, False),
])
def test_every_block_keeps_all_its_keys(B, H, S, D, causal):
    """The splits of a block cover its key tiles exactly once, every split
    has at least one tile, and the item count per head is the sum."""
    splits, items = fa.fa_split_plan(B, H, S, D, causal, SMS)
    assert items == sum(splits)
    for qb, n in enumerate(splits):
        T = _block_tiles(qb, S, causal)
        c = math.ceil(T / n)
        covered = []
        for s in range(n):
            lo, hi = s * c, min(T, (s + 1) * c)
            assert hi > lo
            covered += list(range(lo, hi))
        assert covered == list(range(T))


def test_invalid_sizes_are_rejected():
    lib = fa.library()
    import ctypes
    arr = (ctypes.c_int * 4)()
    assert lib.fa_split_plan(0, 1, 256, 64, 0, SMS, arr, 4, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_split_plan(1, 1, 256, 64, 0, 0, arr, 4, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_split_plan(1, 1, 256, 64, 0, SMS, None, 4, None) == fa.FA_ERR_INVALID_ARG
