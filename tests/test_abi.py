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


def _draft_conf(L, **kw):
    a = dict(U=FAKE, W1=FAKE, W2t=FAKE, dtype=1, anchor=FAKE, bs=4, gamma=7, V=1024, r=32,
             temperature=1.0, seed=0, step=0, tokens=FAKE, logit_x=FAKE, lse=FAKE, h=FAKE, d=64, w=FAKE, b=0.0,
             sts_T=FAKE, conf=FAKE, surv=FAKE, z_logit=None, ws=FAKE, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return L.dspark_draft_confidence_block(*a.values())


def test_draft_confidence_host_validation(L):
    """The fused call checks both calls' arguments before anything runs."""
    assert _draft_conf(L, U=None) == B.DSPARK_EINVAL
    assert _draft_conf(L, gamma=17) == B.DSPARK_EUNSUPPORTED
    assert _draft_conf(L, h=None) == B.DSPARK_EINVAL
    assert _draft_conf(L, surv=None) == B.DSPARK_EINVAL
    assert _draft_conf(L, d=60) == B.DSPARK_EINVAL
    assert _draft_conf(L, d=1 << 17) == B.DSPARK_EUNSUPPORTED
    assert _draft_conf(L, b=float("inf")) == B.DSPARK_EINVAL
    assert _draft_conf(L, z_logit=FAKE + 2) == B.DSPARK_EINVAL
    assert _draft_conf(L, ws=None) == B.DSPARK_EWORKSPACE


def test_other_entry_points_host_validation(L):
    f = FAKE
    # confidence: d not a multiple of 8
    assert L.dspark_confidence(f, f, 1, f, f, f, 0.0, f, 4, 7, 60, 32, 1024, f, f, None, None) == B.DSPARK_EINVAL
    assert L.dspark_confidence(f, f, 1, f, f, f, 0.0, f, 4, 7, 64, 32, 1024, f, f, f + 2, None) == B.DSPARK_EINVAL
    # observability: bad bin count, missing stats, missing workspace
    assert L.dspark_observe(f, None, f, None, 4, 7, 0, f, f, 1 << 20, None) == B.DSPARK_EINVAL
    assert L.dspark_observe(f, None, f, None, 4, 7, 65, f, f, 1 << 20, None) == B.DSPARK_EINVAL
    assert L.dspark_observe(f, None, f, None, 4, 7, 10, None, f, 1 << 20, None) == B.DSPARK_EINVAL
    assert L.dspark_observe(f, None, f, None, 4, 7, 10, f, None, 0, None) == B.DSPARK_EWORKSPACE
    # temperature fit: sizes, grid too long, workspace too small
    assert L.dspark_sts_fit_workspace_bytes(64, 10) == 64 * 3 * 10 * 8
    assert L.dspark_sts_fit_workspace_bytes(0, 10) == 0 and L.dspark_sts_fit_workspace_bytes(8, 65) == 0
    assert L.dspark_sts_fit(f, f, 0, 7, f, 8, 10, f, f, f, 1 << 20, None) == B.DSPARK_EINVAL
    assert L.dspark_sts_fit(f, f, 100, 17, f, 8, 10, f, f, f, 1 << 20, None) == B.DSPARK_EUNSUPPORTED
    assert L.dspark_sts_fit(f, f, 100, 7, f, 2000, 10, f, f, f, 1 << 30, None) == B.DSPARK_EUNSUPPORTED
    assert L.dspark_sts_fit(f, f, 100, 7, f, 8, 10, f, f, f, 16, None) == B.DSPARK_EWORKSPACE
    # schedule: m_max < bs, bad mode, too many slots, no / small / misaligned workspace
    assert L.dspark_schedule(f, 4, 7, f, 3, 0, f, f, f, f, 256, None) == B.DSPARK_EINVAL
    assert L.dspark_schedule(f, 4, 7, f, 64, 5, f, f, f, f, 256, None) == B.DSPARK_EINVAL
    assert L.dspark_schedule(f, 256, 17, f, 9000, 0, f, f, f, f, 256, None) == B.DSPARK_EUNSUPPORTED
    assert L.dspark_schedule(f, 4, 7, f, 64, 0, f, f, f, None, 256, None) == B.DSPARK_EWORKSPACE
    assert L.dspark_schedule(f, 4, 7, f, 64, 0, f, f, f, f, 255, None) == B.DSPARK_EWORKSPACE
    assert L.dspark_schedule(f, 4, 7, f, 64, 0, f, f, f, f + 16, 256, None) == B.DSPARK_EWORKSPACE
    # asynchronous scheduler: no ring, m_max < bs, too many slots, no workspace
    assert L.dspark_schedule_zos_select(f, 4, 7, f, 64, None, 0, f, f, f, 256, None) == B.DSPARK_EINVAL
    assert L.dspark_schedule_zos_select(f, 4, 7, f, 3, f, 0, f, f, f, 256, None) == B.DSPARK_EINVAL
    assert L.dspark_schedule_zos_select(f, 256, 17, f, 9000, f, 0, f, f, f, 256, None) == B.DSPARK_EUNSUPPORTED
    assert L.dspark_schedule_zos_select(f, 4, 7, f, 64, f, 0, f, f, None, 0, None) == B.DSPARK_EWORKSPACE
    assert L.dspark_schedule_zos_budget(f, 4, 7, f, 64, None, 0, f, 256, None) == B.DSPARK_EINVAL
    assert L.dspark_schedule_zos_budget(f, 0, 7, f, 64, f, 0, f, 256, None) == B.DSPARK_EINVAL
    assert L.dspark_schedule_zos_budget(f, 4, 7, f, 64, f + 2, 0, f, 256, None) == B.DSPARK_EINVAL
    assert L.dspark_schedule_zos_budget(f, 4, 7, f, 64, f, 0, None, 0, None) == B.DSPARK_EWORKSPACE
    # pack: negative tier count, missing workspace
    assert L.dspark_pack(None, f, f, 4, 7, f, -1, 64, f, f, f, f, f, f, 1 << 20, None) == B.DSPARK_EINVAL
    assert L.dspark_pack(None, f, f, 4, 7, None, 0, 64, f, f, f, f, f, None, 0, None) == B.DSPARK_EWORKSPACE
    # verify: compact without window, cap-accept without ceiling, bad mode, no source for p_d,
    # misaligned draft logits
    args = [f, 1, f, None, 1, 4, 7, 1024, f, f, f, f, None, None, f, f, f, 32, 1.0, 0, 0, f, f, f, f, 1 << 30, None]
    assert L.dspark_verify(*args) == B.DSPARK_EINVAL
    args[3], args[4], args[23] = f, 2, None
    assert L.dspark_verify(*args) == B.DSPARK_EINVAL
    args[4] = 9
    assert L.dspark_verify(*args) == B.DSPARK_EINVAL
    args[4], args[23] = 1, f
    args[13] = f + 8  # RNN states given, not 16-byte aligned
    assert L.dspark_verify(*args) == B.DSPARK_EINVAL
    args[13] = None
    args[14] = None  # neither draft logits nor U
    assert L.dspark_verify(*args) == B.DSPARK_EINVAL
    args[12] = f + 2  # draft logits given, not 16-byte aligned
    assert L.dspark_verify(*args) == B.DSPARK_EINVAL


def test_rnn_draft_host_validation(L):
    f = FAKE
    base = dict(U=f, W1=f, W2t=f, Wg=f, bg=f, dtype=1, anchor=f, bs=4, gamma=7, V=1024, r=32,
                temperature=ctypes.c_float(1.0), seed=0, step=0, tokens=f, logit_x=f, lse=f, states=f, ws=f,
                ws_bytes=1 << 30, stream=None)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return L.dspark_draft_block_rnn(*a.values())
    assert call(Wg=None) == B.DSPARK_EINVAL
    assert call(bg=None) == B.DSPARK_EINVAL
    assert call(states=None) == B.DSPARK_EINVAL
    assert call(states=f + 4) == B.DSPARK_EINVAL
    assert call(bs=300) == B.DSPARK_EUNSUPPORTED
    assert call(r=48) == B.DSPARK_EUNSUPPORTED
    assert call(ws=None) == B.DSPARK_EWORKSPACE


def test_schedule_pack_host_validation(L):
    f = FAKE
    assert L.dspark_schedule_pack(None, 4, 7, f, 64, 1, f, f, f, f, f, None, 0, 64, f, f, f, f, f, f, 1 << 20,
                                  None) == B.DSPARK_EINVAL
    assert L.dspark_schedule_pack(f, 4, 7, f, 64, 5, f, f, f, f, f, None, 0, 64, f, f, f, f, f, f, 1 << 20,
                                  None) == B.DSPARK_EINVAL          # unknown mode
    assert L.dspark_schedule_pack(f, 4, 7, f, 64, 1, f, f, f, f, f, None, 0, 64, f, f, f, f, f, None, 0,
                                  None) == B.DSPARK_EWORKSPACE
    assert L.dspark_schedule_pack(f, 300, 7, f, 4000, 1, f, f, f, f, f, None, 0, 64, f, f, f, f, f, f, 1 << 20,
                                  None) == B.DSPARK_EUNSUPPORTED


def test_copy_packed_rows_host_validation(L):
    """Bad arguments are refused on the host before any copy is enqueued."""
    f = FAKE
    cu = np.array([0, 3, 3, 9], dtype=np.int32)      # 3 requests: 3, 0, 6 rows
    p = cu.ctypes.data
    assert L.dspark_copy_packed_rows_async(None, f, 64, 3, 8, p, None) == B.DSPARK_EINVAL
    assert L.dspark_copy_packed_rows_async(f, None, 64, 3, 8, p, None) == B.DSPARK_EINVAL
    assert L.dspark_copy_packed_rows_async(f, f, 64, 3, 8, None, None) == B.DSPARK_EINVAL
    assert L.dspark_copy_packed_rows_async(f, f, 0, 3, 8, p, None) == B.DSPARK_EINVAL
    assert L.dspark_copy_packed_rows_async(f, f, 64, 3, 0, p, None) == B.DSPARK_EINVAL
    assert L.dspark_copy_packed_rows_async(f, f, 64, 3, 5, p, None) == B.DSPARK_EINVAL   # 6 rows > 5
    bad = np.array([0, 4, 2, 5], dtype=np.int32)     # decreasing
    assert L.dspark_copy_packed_rows_async(f, f, 64, 3, 8, bad.ctypes.data, None) == B.DSPARK_EINVAL


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


def test_constants_match_the_header_and_the_oracle():
    """The binding's size and chunk constants are the header's; the chunk widths are the ones
    the oracle's draws use (the chunk width fixes which random words a draw consumes)."""
    src = open(HEADER).read()
    defs = {k: int(v) for k, v in re.findall(r"#define\s+(DSPARK_\w+)\s+(\d+)\b", src)}
    for name in ("DSPARK_MAX_BS", "DSPARK_MAX_GAMMA", "DSPARK_CHUNK", "DSPARK_DRAFT_CHUNK"):
        assert getattr(B, name) == defs[name], name
    assert defs["DSPARK_CHUNK"] == O.CHUNK and defs["DSPARK_DRAFT_CHUNK"] == O.DRAFT_CHUNK
    assert defs["DSPARK_MAX_GAMMA"] == O.MAX_GAMMA


def test_obs_structures_match_the_header(tmp_path):
    """The binding's ctypes structures have the C layout (sizes and field offsets)."""
    import ctypes
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = ["steps", "sum_accepted_ceiling", "window_hist", "ceiling_hist", "bin_count", "bin_score_fx",
              "pos_count", "pos_score_fx"]
    src = tmp_path / "layout.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"dspark.h\"\nint main(void){\n"
                   'printf("%zu %zu\\n", sizeof(dspark_obs_stats), sizeof(dspark_obs_summary));\n'
                   + "".join(f'printf("%zu\\n", offsetof(dspark_obs_stats, {f}));\n' for f in fields)
                   + 'printf("%zu %zu\\n", offsetof(dspark_obs_summary, pos_pass_rate), offsetof(dspark_obs_summary, scored));\n'
                   + "return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I" + os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    got = [int(x) for x in out]
    assert got[0] == ctypes.sizeof(B.ObsStats) and got[1] == ctypes.sizeof(B.ObsSummary)
    assert got[2:2 + len(fields)] == [getattr(B.ObsStats, f).offset for f in fields]
    assert got[-2:] == [B.ObsSummary.pos_pass_rate.offset, B.ObsSummary.scored.offset]


def test_obs_report_matches_oracle(L):
    """The host report of the C library on records made from the oracle's observe()."""
    rng = np.random.default_rng(4)
    bs, gamma, M = 32, 7, 12
    st = B.ObsStats()
    recs = []
    for t in range(3):
        surv = I.random_survival(bs, gamma, 50 + t)
        ceiling = rng.integers(0, gamma + 1, bs)
        window = rng.integers(0, gamma + 1, bs)
        acc = np.minimum(ceiling, window)
        recs.append(O.observe(surv, window, acc, ceiling if t != 1 else None, M))
    tot = {k: sum(r[k] for r in recs) for k in recs[0]}
    for k in ("steps", "requests", "sum_window", "sum_accepted", "ceiling_requests", "sum_ceiling",
              "sum_accepted_ceiling"):
        setattr(st, k, int(tot[k]))
    for k in ("window_hist", "accepted_hist", "ceiling_hist"):
        getattr(st, k)[:] = [int(v) for v in tot[k]]
    st.bin_count[:M] = [int(v) for v in tot["bin_count"]]
    st.bin_label[:M] = [int(v) for v in tot["bin_label"]]
    st.bin_score_fx[:M] = [int(round(v * 2.0 ** 32)) for v in tot["bin_score"]]
    st.pos_count[:gamma] = [int(v) for v in tot["pos_count"]]
    st.pos_label[:gamma] = [int(v) for v in tot["pos_label"]]
    st.pos_score_fx[:gamma] = [int(round(v * 2.0 ** 32)) for v in tot["pos_score"]]
    got = B.dspark_obs_report(st, M)
    ref = O.obs_report(tot)
    for k in ("mean_window", "mean_accepted", "mean_ceiling", "utilisation", "ece"):
        assert got[k] == pytest.approx(ref[k], rel=1e-9, abs=1e-9), k
    np.testing.assert_allclose(got["pos_mean_survival"][:gamma], ref["pos_mean_survival"], rtol=1e-9)
    np.testing.assert_allclose(got["pos_pass_rate"][:gamma], ref["pos_pass_rate"], rtol=1e-12)
    assert all(np.isnan(got["pos_pass_rate"][gamma:]))
    assert got["scored"] == int(np.sum(tot["bin_count"]))


def test_stage_ranges_are_inert_by_default():
    """The NVTX stage ranges of step.py cost nothing unless DSPARK_NVTX=1."""
    from speculative_decoding_draft_markov_gb300 import step as S
    ran = []
    with S.stage("x"):
        ran.append(1)
    assert ran == [1] and S._NVTX is False
