"""The C ABI on the CPU: the library builds for sm_103a, loads, exports every entry point
that include/dspark.h declares, rejects bad arguments on the host without touching a GPU,
and its host cost-table builder agrees with the oracle."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

from oracle import dspark_oracle as O
from speculative_decoding_draft_markov_gb300 import binding as B
from speculative_decoding_draft_markov_gb300 import build as BUILD
from speculative_decoding_draft_markov_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


@pytest.fixture(scope="module")
def L():
    BUILD.build()
    return B.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    # the binding wraps every one of them under the same name
    for n in names:
        assert hasattr(B, n), n


def test_status_strings(L):
    for code in range(6):
        assert B.dspark_status_string(code).startswith("DSPARK_")
    assert "UNKNOWN" in B.dspark_status_string(99)


def test_workspace_bytes(L):
    assert B.dspark_workspace_bytes(0, 7, 1024) == 0
    assert B.dspark_workspace_bytes(257, 7, 1024) == 0
    assert B.dspark_workspace_bytes(4, 17, 1024) == 0
    n = B.dspark_workspace_bytes(256, 7, 151936)
    nchunks = (151936 + 127) // 128
    assert n >= 256 * nchunks * 8 + 256 * 8 * 16 + 256 * 16
    assert n % 256 == 0


FAKE = 1 << 20  # a non-null, aligned host address the library never dereferences on these paths


def _draft(L, **kw):
    a = dict(U=FAKE, W1=FAKE, W2t=FAKE, dtype=1, anchor=FAKE, bs=4, gamma=7, V=1024, r=32,
             temperature=1.0, seed=0, step=0, tokens=FAKE, logit_x=FAKE, lse=FAKE, ws=FAKE,
             ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return L.dspark_draft_block(*a.values())


def test_draft_host_validation(L):
    assert _draft(L, U=None) == B.DSPARK_EINVAL
    assert _draft(L, bs=0) == B.DSPARK_EINVAL
    assert _draft(L, bs=300) == B.DSPARK_EUNSUPPORTED
    assert _draft(L, gamma=17) == B.DSPARK_EUNSUPPORTED
    assert _draft(L, V=1001) == B.DSPARK_EINVAL
    assert _draft(L, r=48) == B.DSPARK_EUNSUPPORTED
    assert _draft(L, dtype=7) == B.DSPARK_EINVAL
    assert _draft(L, temperature=-1.0) == B.DSPARK_EINVAL
    assert _draft(L, temperature=float("nan")) == B.DSPARK_EINVAL
    assert _draft(L, U=FAKE + 2) == B.DSPARK_EINVAL
    assert _draft(L, ws=None) == B.DSPARK_EWORKSPACE
    assert _draft(L, ws_bytes=16) == B.DSPARK_EWORKSPACE


def test_other_entry_points_host_validation(L):
    f = FAKE
    # confidence: d not a multiple of 8
    assert L.dspark_confidence(f, f, 1, f, f, f, 0.0, f, 4, 7, 60, 32, 1024, f, f, None) == B.DSPARK_EINVAL
    # schedule: m_max < bs, bad mode, too many slots
    assert L.dspark_schedule(f, 4, 7, f, 3, 0, f, f, f, None) == B.DSPARK_EINVAL
    assert L.dspark_schedule(f, 4, 7, f, 64, 5, f, f, f, None) == B.DSPARK_EINVAL
    assert L.dspark_schedule(f, 256, 17, f, 9000, 0, f, f, f, None) == B.DSPARK_EUNSUPPORTED
    # asynchronous scheduler: no ring, m_max < bs, too many slots
    assert L.dspark_schedule_zos_select(f, 4, 7, f, 64, None, 0, f, f, None) == B.DSPARK_EINVAL
    assert L.dspark_schedule_zos_select(f, 4, 7, f, 3, f, 0, f, f, None) == B.DSPARK_EINVAL
    assert L.dspark_schedule_zos_select(f, 256, 17, f, 9000, f, 0, f, f, None) == B.DSPARK_EUNSUPPORTED
    assert L.dspark_schedule_zos_budget(f, 4, 7, f, 64, None, 0, None) == B.DSPARK_EINVAL
    assert L.dspark_schedule_zos_budget(f, 0, 7, f, 64, f, 0, None) == B.DSPARK_EINVAL
    assert L.dspark_schedule_zos_budget(f, 4, 7, f, 64, f + 2, 0, None) == B.DSPARK_EINVAL
    # pack: negative tier count, missing workspace
    assert L.dspark_pack(None, f, f, 4, 7, f, -1, 64, f, f, f, f, f, f, 1 << 20, None) == B.DSPARK_EINVAL
    assert L.dspark_pack(None, f, f, 4, 7, None, 0, 64, f, f, f, f, f, None, 0, None) == B.DSPARK_EWORKSPACE
    # verify: compact without window, cap-accept without ceiling, bad mode, no source for p_d,
    # misaligned draft logits
    args = [f, 1, f, None, 1, 4, 7, 1024, f, f, f, f, None, f, f, f, 32, 1.0, 0, 0, f, f, f, f, 1 << 30, None]
    assert L.dspark_verify(*args) == B.DSPARK_EINVAL
    args[3], args[4], args[22] = f, 2, None
    assert L.dspark_verify(*args) == B.DSPARK_EINVAL
    args[4] = 9
    assert L.dspark_verify(*args) == B.DSPARK_EINVAL
    args[4], args[22] = 1, f
    args[13] = None  # neither draft logits nor U
    assert L.dspark_verify(*args) == B.DSPARK_EINVAL
    args[12] = f + 2  # draft logits given, not 16-byte aligned
    assert L.dspark_verify(*args) == B.DSPARK_EINVAL


def test_build_sps_matches_oracle(L):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "tier_padding.json")))
    rng = np.random.default_rng(0)
    for tiers in ([], list(range(16, 513, 16)), [3, 7, 8, 100], [8, 16, 24]):
        m_max = 512 if tiers != [8, 16, 24] else 40
        T = 5.0 + 0.01 * np.arange(m_max + 1) + rng.normal(0, 0.05, m_max + 1)
        got = B.dspark_build_sps(T, np.array(tiers, dtype=np.int32))
        np.testing.assert_array_equal(got, O.build_sps(T, tiers))
    tiers = np.arange(g["tiers_every"], g["tier_max"] + 1, g["tiers_every"], dtype=np.int32)
    sps = B.dspark_build_sps(5.0 + 0.01 * np.arange(g["tier_max"] + 1), tiers)
    for case in g["cases"]:
        assert sps[case["total"]] == sps[case["tier"]]
    for wl in I.WORKLOADS.values():
        np.testing.assert_array_equal(B.dspark_build_sps(I.cost_curve_ms(wl), I.tiers_for(wl)),
                                      O.build_sps(I.cost_curve_ms(wl), I.tiers_for(wl)))
    with pytest.raises(B.DSparkError):
        B.dspark_build_sps(np.array([1.0, -1.0]), np.zeros(0, np.int32))
    with pytest.raises(B.DSparkError):
        B.dspark_build_sps(np.ones(10), np.array([4, 4], np.int32))
