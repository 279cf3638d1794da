"""The split-count cost model (host logic, no GPU): attn_fwd's own split and attn_fwd_splitkv's
default, through the test hook that takes the device's SM count and cluster capacity as
arguments (152 SMs and 76 / 48 / 36 clusters of 2 / 3 / 4 CTAs stand for a GB300)."""
import ctypes

import pytest

from exact_attention_forward_attn_gb300 import _lib, build
from exact_attention_forward_attn_gb300 import workloads as wl

SMS = 152
FIT = (76, 48, 36)
UNLIMITED = 2 ** 62
FWD_SCRATCH = 64 << 20  # one slot of attn_fwd's own split scratch


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _choice(lib, B, Hq, N, D, causal, cluster_only, max_ws=UNLIMITED, sms=SMS, fit=FIT):
    return lib.attn_fwd_test_split_choice(B, Hq, N, D, int(causal), sms,
                                          (ctypes.c_int * 3)(*fit), int(cluster_only), max_ws)


@pytest.mark.parametrize("w", [wl.TINY_NONCAUSAL, wl.TINY_CAUSAL, wl.GQA4_CAUSAL, wl.GQA8_CAUSAL,
                               wl.MHA, wl.MQA] + [wl.LONG[n] for n in sorted(wl.LONG)],
                         ids=lambda w: w.name)
def test_the_five_configurations_run_the_single_pass(w, lib):
    assert _choice(lib, w.B, w.Hq, w.N, w.D, w.causal, True) == 1
    assert _choice(lib, w.B, w.Hq, w.N, w.D, w.causal, False, max_ws=FWD_SCRATCH) == 1
    assert _choice(lib, w.B, w.Hq, w.N, w.D, w.causal, False) == 1


def test_few_heads_over_long_keys_split(lib):
    # two heads of 4096 rows: 16 pairs of Q tiles per head on 152 SMs; by the model's constants
    # 4 splits merged inside clusters (17.5 + 0.5 + 8 x 1.2 = 27.6 us) beat the single pass on one
    # Q tile per CTA (10 + 0.5 + 32 x 1.0 = 42.5 us) and 2 or 3 splits (37.2, 31.2 us)
    w = wl.FEWHEADS
    assert _choice(lib, w.B, w.Hq, w.N, w.D, w.causal, True) == 4
    assert _choice(lib, w.B, w.Hq, w.N, w.D, w.causal, False) == 4
    # causal few heads: the persistent split kernel's balanced claims win (measured 72 against 95
    # us at four heads of 8192 rows); attn_fwd takes that path through its scratch slots, except
    # under graph capture (cluster splits only: 128 pairs are more clusters than fit at once)
    assert _choice(lib, 1, 4, 8192, 128, True, False) >= 2
    assert _choice(lib, 1, 4, 8192, 128, True, False, max_ws=FWD_SCRATCH) >= 2
    assert _choice(lib, 1, 4, 8192, 128, True, True) == 1


def test_attn_fwd_splits_only_into_clusters_that_fit(lib):
    for B, Hq, N, D, c in [(1, 1, 8192, 128, False), (1, 2, 4096, 64, True), (1, 1, 16384, 128, True)]:
        n = _choice(lib, B, Hq, N, D, c, True)
        assert 2 <= n <= 4
        assert _choice(lib, B, Hq, N, D, c, True, fit=(0, 0, 0)) == 1
    # only 4-CTA clusters fit: a 2- or 3-way split is never chosen
    for N in (2048, 4096, 8192, 16384):
        assert _choice(lib, 1, 1, N, 128, False, True, fit=(0, 0, 64)) in (1, 4)


def test_many_query_tiles_are_never_split(lib):
    # at least twice as many Q-tile pairs as SMs
    for B, Hq, N in [(1, 2, 65536), (1, 1, 131072), (4, 32, 2048), (1, 64, 4096)]:
        assert _choice(lib, B, Hq, N, 128, True, False) == 1
        assert _choice(lib, B, Hq, N, 128, False, True) == 1


def test_default_respects_a_workspace_limit(lib):
    for B, Hq, N, D, c in [(1, 4, 8192, 128, True), (1, 1, 16384, 128, True), (1, 2, 16384, 64, True),
                           (2, 1, 8192, 128, False), (1, 8, 4096, 128, True)]:
        for limit in (0, 8 << 20, 32 << 20, 64 << 20, UNLIMITED):
            n = _choice(lib, B, Hq, N, D, c, False, max_ws=limit)
            assert n >= 1
            assert lib.attn_fwd_splitkv_workspace_bytes(B, Hq, N, D, n) <= limit


def test_attn_fwd_scratch_limit_caps_the_split(lib):
    # one causal head of 65536 rows: 4 splits need 135 MB of partials, beyond a 64 MiB slot
    n = _choice(lib, 1, 1, 65536, 128, False, False, max_ws=FWD_SCRATCH)
    assert lib.attn_fwd_splitkv_workspace_bytes(1, 1, 65536, 128, n) <= FWD_SCRATCH


def test_single_query_tile_and_wide_heads(lib):
    assert _choice(lib, 1, 1, 128, 128, False, False) == 1  # one key tile: nothing to split
    assert _choice(lib, 1, 1, 8192, 256, False, False) == 1  # D > 128: no split form
    assert _choice(lib, 1, 1, 8192, 256, False, True) == 1


def test_invalid_arguments(lib):
    assert _choice(lib, 0, 1, 1024, 128, False, True) == -2
    assert _choice(lib, 1, 1, 1024, 100, False, True) == -2
    assert _choice(lib, 1, 1, 1024, 128, False, True, sms=0) == -2
    assert _choice(lib, 1, 1, 1024, 128, False, False, max_ws=-1) == -2
