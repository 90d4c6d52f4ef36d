"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Every output buffer is pre-filled with the same sentinel on both sides and
compared bit for bit over its whole extent, so rows the definition does not
name must stay untouched. Layout, payload and scale bytes must be identical;
the combine must equal the oracle's fp32-FMA twin bit for bit and lie within
one bf16 ulp of the fp64 sum (plus the fp32 accumulation floor K*2^-24*sum|w*y|).
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import DEV, bf16_dev, bf16_ulp, bits_equal, first_mismatch, to_dev, to_host

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def assert_same(name, got, want):
    assert bits_equal(got, want), f"{name}: first differing byte / count {first_mismatch(got, want)}"


def compact_both(mp, ref, x, ids, w, H, K, E, L, b, g, fmt, n_live=None, ldx=None, with_rw=True):
    T = ids.shape[0]
    G = H // g
    ldx = H if ldx is None else ldx
    bound = ref.compact_bound(T * K, L, b)
    r = {"xq": np.full((bound, H), 0xEE, np.uint8)}
    r["sc"], ld = ref.scale_buffer(fmt, bound, G, fill=0xA5)
    r["mi"] = np.full(bound, -7, np.int32)
    r["s2d"] = np.full((T, K), -9, np.int32)
    r["counts"] = np.full(L, -5, np.int32)
    r["starts"] = np.full(L, -5, np.int32)
    r["psum"] = np.full(L, -5, np.int32)
    r["total"] = np.full(1, -3, np.int32)
    r["rw"] = np.full(bound, np.nan, np.float32) if with_rw else None
    d = {k: (to_dev(v.copy()) if v is not None else None) for k, v in r.items()}
    nl = T if n_live is None else n_live
    st_ref = ref.dispatch_compact(x, T, nl, H, ids, w, K, L, b, g, fmt, r["xq"], r["sc"], ld,
                                  r["mi"], bound, r["s2d"], r["counts"], r["starts"], r["psum"],
                                  r["total"], r["rw"], ldx=ldx)
    ws = mp.Workspace(T, K, L, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    nld = None if n_live is None else torch.tensor([n_live], dtype=torch.int32, device=DEV)
    code = mp.moe_dispatch_compact(bf16_dev(x), ldx, T, nld, H, to_dev(ids), to_dev(w), K, E, L, b,
                                   g, fmt, d["xq"], d["sc"], ld, d["mi"], bound, d["s2d"],
                                   d["counts"], d["starts"], d["psum"], d["total"], d["rw"],
                                   ws.buf, ws.nbytes, status)
    assert code == mp.MOE_OK
    torch.cuda.synchronize()
    for k, v in r.items():
        if v is not None:
            assert_same(k, to_host(d[k], v), v)
    assert int(status.item()) == st_ref
    return r, d, ws


def masked_both(mp, ref, x, ids, w, H, K, E, L, cap, g, fmt, n_live=None, psum_align=128):
    """Masked dispatch on both sides; psum_align None leaves the psum output out."""
    T = ids.shape[0]
    G = H // g
    r = {"xq": np.full((L * cap, H), 0xEE, np.uint8)}
    r["sc"], ld = ref.scale_buffer(fmt, L * cap, G, fill=0xA5, blocks=L)
    r["mm"] = np.full(L, -5, np.int32)
    r["s2d"] = np.full((T, K), -9, np.int32)
    r["rw"] = np.full(L * cap, np.nan, np.float32)
    if psum_align is not None:
        r["psum"] = np.full(L, -5, np.int32)
    d = {k: to_dev(v.copy()) for k, v in r.items()}
    nl = T if n_live is None else n_live
    st_ref = ref.dispatch_masked(x, T, nl, H, ids, w, K, L, cap, g, fmt, r["xq"], r["sc"], ld,
                                 r["mm"], r["s2d"], r["rw"], psum=r.get("psum"),
                                 psum_align=psum_align or 1)
    ws = mp.Workspace(T, K, L, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    nld = None if n_live is None else torch.tensor([n_live], dtype=torch.int32, device=DEV)
    code = mp.moe_dispatch_masked(bf16_dev(x), H, T, nld, H, to_dev(ids), to_dev(w), K, E, L, cap,
                                  g, fmt, d["xq"], d["sc"], ld, d["mm"], d["s2d"], d["rw"],
                                  d.get("psum"), psum_align or 1, ws.buf, ws.nbytes, status)
    assert code == mp.MOE_OK
    torch.cuda.synchronize()
    for k, v in r.items():
        assert_same(k, to_host(d[k], v), v)
    assert int(status.item()) == st_ref
    return r, d, status


def check_combine(mp, ref, y, s2d, w, H, n_live=None):
    T, K = s2d.shape
    R = y.shape[0]
    want32 = ref.combine_f32(y, s2d, w, T, K, H)
    want64, mass = ref.combine_f64(y, s2d, w, T, K, H)
    out = torch.full((T, H), -12345.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    nld = None if n_live is None else torch.tensor([n_live], dtype=torch.int32, device=DEV)
    code = mp.moe_combine(bf16_dev(y), H, R, to_dev(s2d), None if w is None else to_dev(w), T, nld,
                          K, H, out, status)
    assert code == mp.MOE_OK
    torch.cuda.synchronize()
    got = to_host(out.view(torch.int16), want32)
    n = T if n_live is None else n_live
    assert_same("combine vs fp32-FMA twin", got[:n], want32[:n])
    if n < T:
        sentinel = to_host(torch.full((1,), -12345.0, dtype=torch.bfloat16).view(torch.int16), np.zeros(1, np.uint16))[0]
        assert (got[n:] == sentinel).all(), "rows of non-live tokens untouched"
    gf = synth.from_bf16_bits(got[:n]).astype(np.float64)
    err = np.abs(gf - want64[:n])
    tol = bf16_ulp(want64[:n]) + K * 2.0 ** -24 * mass[:n]
    assert (err <= tol).all(), f"max err/tol {np.max(err / tol)}"
    assert int(status.item()) == 0
    return got


# ---------------------------------------------------------------------------
# quantisation
# ---------------------------------------------------------------------------

def test_e4m3_convert_exhaustive_via_quant_group(dev, ref):
    """Every finite bf16 value x, scaled by 2^-e for several group exponents e:
    each group of 32 holds one element 448*2^e that fixes the exponent and 31
    test values with |x| <= 448*2^e. GPU bytes must equal the oracle's."""
    H, g = 7168, 32
    allb = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    vals = synth.from_bf16_bits(allb)
    finite = np.isfinite(vals)
    for e in (-42, -20, -6, 0, 3, 9, 60, 119):
        amax = np.float32(448.0 * 2.0 ** e)
        amax_b = synth.to_bf16_bits(np.array([amax], np.float32))[0]
        test = allb[finite & (np.abs(vals) <= amax)]
        ngroups = -(-test.size // 31)
        pad = np.resize(test, ngroups * 31) if test.size else np.zeros(31, np.uint16)
        groups = np.concatenate([np.full((ngroups, 1), amax_b, np.uint16), pad.reshape(ngroups, 31)], axis=1)
        per_row = H // g
        nrows = -(-ngroups // per_row)
        rows = np.zeros((nrows * per_row, g), np.uint16)
        rows[:] = amax_b
        rows[:ngroups] = groups
        x = rows.reshape(nrows, H)
        rxq = np.full((nrows, H), 0xEE, np.uint8)
        rsc, ld = ref.scale_buffer("u8", nrows, H // g)
        ref.quant_group(x, nrows, nrows, H, g, "u8", rxq, rsc, ld)
        assert (rsc == 127 + e).all()
        out = dev.quant_group(bf16_dev(x), group_size=g, scale_fmt="u8")
        torch.cuda.synchronize()
        assert_same(f"xq e={e}", to_host(out["xq"], rxq), rxq)
        assert_same(f"scales e={e}", to_host(out["scales"], rsc), rsc)


@pytest.mark.parametrize("fmt,g,T,H", [("packed", 128, 50, 640), ("u8", 128, 33, 7168),
                                       ("f32pow2", 128, 17, 1152), ("u8", 32, 5, 224),
                                       ("packed", 128, 257, 7168), ("f32", 128, 33, 7168),
                                       ("f32", 128, 5, 640), ("mx", 32, 21, 7168),
                                       ("mx", 32, 3, 224)])
def test_quant_group_formats(dev, ref, fmt, g, T, H):
    rng = np.random.default_rng(T + H)
    x = synth.normal_bf16(rng, (T, H), outlier_frac=0.02)
    x[0, :g] = 0                     # an all-zero group
    G = H // g
    rxq = np.full((T, H), 0xEE, np.uint8)
    rsc, ld = ref.scale_buffer(fmt, T, G, fill=0x5A)
    ref.quant_group(x, T, T, H, g, fmt, rxq, rsc, ld)
    dxq, dsc = to_dev(rxq.copy()), to_dev(rsc.copy())
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert dev.moe_quant_group(bf16_dev(x), H, T, None, H, g, fmt, dxq, dsc, ld, st) == 0
    torch.cuda.synchronize()
    assert_same("xq", to_host(dxq, rxq), rxq)
    assert_same("scales", to_host(dsc, rsc), rsc)


def test_mxfp8_sparse_live_rows_full_size(dev, ref):
    """24576-row receive buffer, 112 live rows, the rest NaN/Inf garbage: only
    live rows are read and written; group-32 e8m0, 224 scales per row."""
    d = synth.mxfp8(0)
    c = d["cfg"]
    T_cap, n, H, g = c["T_cap"], c["n_live"], c["H"], c["g"]
    assert H // g == 224
    rxq = np.full((T_cap, H), 0xEE, np.uint8)
    rsc, ld = ref.scale_buffer("u8", T_cap, H // g)
    assert ref.quant_group(d["x"], T_cap, n, H, g, "u8", rxq, rsc, ld) == 0
    dxq, dsc = to_dev(rxq), to_dev(rsc)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    nl = torch.tensor([n], dtype=torch.int32, device=DEV)
    assert dev.moe_quant_group(bf16_dev(d["x"]), H, T_cap, nl, H, g, "u8", dxq, dsc, ld, st) == 0
    torch.cuda.synchronize()
    assert_same("xq", to_host(dxq, rxq), rxq)
    assert_same("scales", to_host(dsc, rsc), rsc)
    assert int(st.item()) == 0
    # empty live batch: nothing written
    nl.zero_()
    before = dxq.clone()
    assert dev.moe_quant_group(bf16_dev(d["x"]), H, T_cap, nl, H, g, "u8", dxq, dsc, ld, st) == 0
    torch.cuda.synchronize()
    assert torch.equal(before, dxq)
    # empty tensor API: scale shape (0, 224)
    out = dev.quant_group(torch.empty((0, H), dtype=torch.bfloat16, device=DEV), group_size=32, scale_fmt="u8")
    assert tuple(out["scales"].shape) == (0, 224) and out["scales"].dtype == torch.uint8
    # live count above the buffer: clamped to the buffer, flagged
    x2 = synth.normal_bf16(np.random.default_rng(1), (64, H))
    st.zero_()
    small_q = torch.empty((64, H), dtype=torch.uint8, device=DEV)
    small_s = torch.empty((64, H // g), dtype=torch.uint8, device=DEV)
    nl.fill_(65)
    assert dev.moe_quant_group(bf16_dev(x2), H, 64, nl, H, g, "u8", small_q, small_s, H // g, st) == 0
    assert dev.moe_status_sync(st) == dev.MOE_ERR_LIVE_OVERFLOW


# ---------------------------------------------------------------------------
# compact dispatch
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("fmt", ["packed", "u8", "f32pow2"])
def test_dispatch_compact_tiny(dev, ref, seed, fmt):
    d = synth.tiny(seed)
    c = d["cfg"]
    compact_both(dev, ref, d["x"], d["topk_ids"], d["topk_weights"], c["H"], c["K"], c["E"], c["L"],
                 c["block_e"], c["g"], fmt)


@pytest.mark.parametrize("T", [203, 613])   # 1624 slots: one-launch path; 4904: two-launch path
@pytest.mark.parametrize("fmt", ["packed", "u8", "f32pow2", "f32"])
def test_dispatch_compact_tiles_and_ragged_tail(dev, ref, fmt, T):
    d = synth.prefill(1, T=T, H=1536)
    compact_both(dev, ref, d["x"], d["topk_ids"], d["topk_weights"], 1536, 8, 256, 256, 128, 128, fmt)


def test_dispatch_compact_nondividing_groups_and_dropped(dev, ref):
    """H = 640 (5 groups: the last packed word is half padding), 40 experts of
    which 20 are local, block_e = 16."""
    rng = np.random.default_rng(3)
    T, K, H = 97, 4, 640
    x = synth.normal_bf16(rng, (T, H))
    ids = synth.uniform_topk(rng, T, 40, K)
    ids[5, 0] = -1
    w = synth.softmax_weights(rng, T, K)
    for fmt in ("packed", "u8"):
        compact_both(dev, ref, x, ids, w, H, K, 40, 20, 16, 128, fmt)


@pytest.mark.parametrize("L", [32, 2])
def test_dispatch_compact_sparse_two_launch(dev, ref, L):
    """Two-launch compact dispatch where many tokens have no local expert
    (top-8 over 256 experts with L local: ~34% of tokens for L = 32, ~94% for
    L = 2). Such tokens are dropped from the scatter's walk; a CTA may be left
    with only its early-staged tokens, or none with a kept slot."""
    rng = np.random.default_rng(100 + L)
    T, K, H = 700, 8, 1024
    x = synth.normal_bf16(rng, (T, H))
    ids = synth.uniform_topk(rng, T, 256, K)
    w = synth.softmax_weights(rng, T, K)
    for fmt in ("packed", "u8"):
        compact_both(dev, ref, x, ids, w, H, K, 256, L, 128, 128, fmt)


def test_dispatch_compact_live_tokens_and_stride(dev, ref):
    rng = np.random.default_rng(4)
    T, K, H, ldx = 200, 8, 1024, 1088
    xf = synth.normal_bf16(rng, (T, ldx))
    xf[150:] = synth.garbage_bf16_rows(T - 150, ldx)
    ids = synth.uniform_topk(rng, T, 64, K)
    ids[150:] = 0x7FFFFFF0          # never read
    w = synth.softmax_weights(rng, T, K)
    r, d, _ = compact_both(dev, ref, xf, ids, w, H, K, 64, 64, 128, 128, "packed", n_live=150, ldx=ldx)
    assert (r["s2d"][150:] == -1).all()


@pytest.mark.parametrize("T,K,L,H", [(4096, 8, 256, 128), (40000, 8, 300, 128), (1, 1, 1, 128),
                                     (3, 2, 1024, 128), (1000, 16, 7, 256)])
def test_dispatch_compact_chunking(dev, ref, T, K, L, H):
    """Route-plan chunk sizes S = 1, 4, 16 and 64 (up to 20 chunks), one CTA, L = 1024."""
    rng = np.random.default_rng(T + L)
    x = synth.normal_bf16(rng, (T, H))
    E = max(L, 2 * K)
    ids = synth.zipf_topk(rng, T, E, K, n_empty=min(12, E - K)) if T > 1 else synth.uniform_topk(rng, T, E, K)
    w = synth.softmax_weights(rng, T, K)
    compact_both(dev, ref, x, ids, w, H, K, E, L, 128, 128, "packed")


def test_dispatch_compact_degenerate(dev, ref):
    rng = np.random.default_rng(6)
    H = 256
    x = synth.normal_bf16(rng, (64, H))
    w = np.ones((64, 4), np.float32)
    compact_both(dev, ref, x, np.full((64, 4), -1, np.int32), w, H, 4, 8, 8, 128, 128, "packed")  # all dropped
    compact_both(dev, ref, x, np.full((64, 4), 3, np.int32), w, H, 4, 8, 8, 128, 128, "u8")      # one hot expert
    compact_both(dev, ref, x[:0], np.zeros((0, 4), np.int32), w[:0], H, 4, 8, 8, 128, 128, "packed")  # T = 0


@pytest.mark.parametrize("fmt", ["u8", "mx"])
def test_dispatch_compact_mxfp8_group32(dev, ref, fmt):
    d = synth.mxfp8(2, T_cap=112, n_live=112)
    compact_both(dev, ref, d["x"], d["topk_ids"], d["topk_weights"], 7168, 8, 256, 256, 128, 32, fmt)


# ---------------------------------------------------------------------------
# masked dispatch
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("fmt", ["packed", "u8", "f32"])
def test_dispatch_masked_decode(dev, ref, seed, fmt):
    d = synth.decode(seed)
    c = d["cfg"]
    assert ref.should_use_masked(c["E"], c["L"])
    masked_both(dev, ref, d["x"], d["topk_ids"], d["topk_weights"], c["H"], c["K"], c["E"], c["L"],
                c["cap"], c["g"], fmt)


@pytest.mark.parametrize("fmt", ["packed", "u8", "f32"])
def test_dispatch_masked_two_launch_path(dev, ref, fmt):
    """T*K = 5600 slots (> 2048): route-plan launch + scatter launch."""
    d = synth.decode(5, T=700)
    x = d["x"][:, :1024].copy()
    masked_both(dev, ref, x, d["topk_ids"], d["topk_weights"], 1024, 8, 256, 32, 128, 128, fmt)


def test_dispatch_masked_overflow_two_launch_path(dev, ref):
    rng = np.random.default_rng(18)
    T, K, H = 600, 8, 256
    x = synth.normal_bf16(rng, (T, H))
    ids = synth.uniform_topk(rng, T, 16, K)      # ~300 slots per local expert
    w = synth.softmax_weights(rng, T, K)
    r, d, status = masked_both(dev, ref, x, ids, w, H, K, 16, 8, 256, 128, "packed")
    assert dev.moe_status_sync(status) == dev.MOE_ERR_OVERFLOW


def test_dispatch_masked_overflow_fails_fast(dev, ref):
    rng = np.random.default_rng(8)
    T, K, H = 64, 8, 512
    x = synth.normal_bf16(rng, (T, H))
    ids = synth.uniform_topk(rng, T, 8, K)       # ~64 slots per local expert
    w = synth.softmax_weights(rng, T, K)
    r, d, status = masked_both(dev, ref, x, ids, w, H, K, 8, 4, 40, 128, "packed")
    assert dev.moe_status_sync(status) == dev.MOE_ERR_OVERFLOW
    masked_both(dev, ref, x, ids, w, H, K, 8, 4, 64, 128, "f32pow2")   # exactly at capacity


def test_dispatch_masked_live_tokens(dev, ref):
    rng = np.random.default_rng(9)
    T, K, H = 96, 8, 1024
    x = synth.normal_bf16(rng, (T, H))
    x[70:] = synth.garbage_bf16_rows(T - 70, H)
    ids = synth.uniform_topk(rng, T, 128, K)
    w = synth.softmax_weights(rng, T, K)
    masked_both(dev, ref, x, ids, w, H, K, 128, 16, 64, 128, "packed", n_live=70)


# ---------------------------------------------------------------------------
# combine
# ---------------------------------------------------------------------------

# K selects the row batch of the combine: ceil(K / ceil(K/4)) rows in flight,
# so 1..4 run one batch, 5..8 two equal ones (3+3, 4+4, 3+2, 4+3), 9..12 three
@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 13, 32])
def test_combine_random_rows(dev, ref, K):
    rng = np.random.default_rng(K)
    T, H, R = 77, 1536, 500
    y = synth.normal_bf16(rng, (R, H))
    s2d = rng.integers(-1, R, size=(T, K)).astype(np.int32)
    s2d[3] = -1
    w = synth.softmax_weights(rng, T, K)
    check_combine(dev, ref, y, s2d, w, H)
    check_combine(dev, ref, y, s2d, None, H)


def test_combine_live_tokens_and_bad_index(dev, ref):
    rng = np.random.default_rng(12)
    T, K, H, R = 40, 8, 512, 100
    y = synth.normal_bf16(rng, (R, H))
    s2d = rng.integers(-1, R, size=(T, K)).astype(np.int32)
    w = synth.softmax_weights(rng, T, K)
    check_combine(dev, ref, y, s2d, w, H, n_live=25)
    bad = s2d.copy()
    bad[2, 1] = R + 7
    out = torch.zeros((T, H), dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert dev.moe_combine(bf16_dev(y), H, R, to_dev(bad), to_dev(w), T, None, K, H, out, st) == 0
    assert dev.moe_status_sync(st) == dev.MOE_ERR_BAD_LAYOUT
    fixed = bad.copy()
    fixed[2, 1] = -1
    want = ref.combine_f32(y, fixed, w, T, K, H)
    assert_same("combine skipping the bad slot", to_host(out.view(torch.int16), want), want)


def test_dispatch_then_combine_masked_equals_compact(dev, ref):
    """PR #33128 test idea on the GPU: expert outputs that depend only on
    (expert, token) give bit-identical combines in both layouts."""
    d = synth.decode(1, T=128)
    c = d["cfg"]
    T, K, E, L, cap, H = 128, 8, 256, 32, 128, 1024
    x = d["x"][:, :H].copy()
    ids, w = d["topk_ids"], d["topk_weights"]
    rc, dc, _ = compact_both(dev, ref, x, ids, w, H, K, E, L, 128, 128, "packed")
    rm, dm, _ = masked_both(dev, ref, x, ids, w, H, K, E, L, cap, 128, "packed")
    rng = np.random.default_rng(5)
    table = synth.normal_bf16(rng, (L, T, H))
    yc = np.zeros((rc["xq"].shape[0], H), np.uint16)
    ym = np.zeros((L * cap, H), np.uint16)
    flat = ids.reshape(-1)
    for a in range(T * K):
        e = flat[a]
        if 0 <= e < L:
            yc[rc["s2d"].reshape(-1)[a]] = table[e, a // K]
            ym[rm["s2d"].reshape(-1)[a]] = table[e, a // K]
    oc = check_combine(dev, ref, yc, rc["s2d"], w, H)
    om = check_combine(dev, ref, ym, rm["s2d"], w, H)
    assert np.array_equal(oc, om)


# ---------------------------------------------------------------------------
# repack
# ---------------------------------------------------------------------------

def build_layout(counts, align):
    starts, psum, prev = [], [], 0
    for cnt in counts:
        st = -(-prev // align) * align
        starts.append(st)
        psum.append(st + cnt)
        prev = st + cnt
    return np.array(psum, np.int32), starts, max(-(-prev // align) * align, 1)


def repack_both(dev, ref, exp, eb, H, psum, L, align, cap, fmt=None, g=128, exp_sc=None, ld_es=0,
                weights=None):
    R = exp.shape[0]
    G = H // g
    slab = np.full((L * cap, H * eb), 0xEE, np.uint8)
    mm = np.full(L, -1, np.int32)
    if exp_sc is not None:
        ssc, ld_ss = ref.scale_buffer(fmt, L * cap, G, fill=0x3C, blocks=L)
    else:
        ssc, ld_ss = None, 0
    st_ref = ref.expand_to_slab(exp, eb, H, R, exp_sc, ld_es, psum, L, align, cap, fmt or "u8", g,
                                slab, ssc, ld_ss, mm)
    d_slab, d_mm = to_dev(np.full_like(slab, 0xEE)), to_dev(np.full_like(mm, -1))
    d_ssc = to_dev(ref.scale_buffer(fmt, L * cap, G, fill=0x3C, blocks=L)[0]) if exp_sc is not None else None
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert dev.moe_expand_to_slab(to_dev(exp), eb, H, R, to_dev(exp_sc) if exp_sc is not None else None,
                                  ld_es, to_dev(psum), L, align, cap, fmt or "u8", g, d_slab, d_ssc,
                                  ld_ss, d_mm, st) == 0
    torch.cuda.synchronize()
    assert_same("slab", to_host(d_slab, slab), slab)
    assert_same("masked_m", to_host(d_mm, mm), mm)
    if ssc is not None:
        assert_same("slab scales", to_host(d_ssc, ssc), ssc)
    assert int(st.item()) == st_ref
    # back to the expanded layout
    back = np.full_like(exp, 0xDD)
    mi = np.full(R, 77, np.int32)
    bsc = ref.scale_buffer(fmt, R, G, fill=0x11)[0] if exp_sc is not None else None
    st2_ref = ref.expand_from_slab(slab, eb, H, ssc, ld_ss, psum, L, align, cap, fmt or "u8", g,
                                   weights, back, R, bsc, ld_es, mi)
    d_back, d_mi = to_dev(np.full_like(exp, 0xDD)), to_dev(np.full(R, 77, np.int32))
    d_bsc = to_dev(ref.scale_buffer(fmt, R, G, fill=0x11)[0]) if exp_sc is not None else None
    st.zero_()
    assert dev.moe_expand_from_slab(d_slab, eb, H, d_ssc, ld_ss, to_dev(psum), L, align, cap,
                                    fmt or "u8", g, to_dev(weights) if weights is not None else None,
                                    d_back, R, d_bsc, ld_es, d_mi, st) == 0
    torch.cuda.synchronize()
    assert_same("expanded", to_host(d_back, back), back)
    assert_same("m_indices", to_host(d_mi, mi), mi)
    if bsc is not None:
        assert_same("expanded scales", to_host(d_bsc, bsc), bsc)
    assert int(st.item()) == st2_ref
    return st_ref, slab, back


@pytest.mark.parametrize("counts", [[3, 0, 5, 1], [0, 0, 0, 0], [0, 17, 0, 0], [8, 8, 8, 8], [1, 0, 0, 9]])
@pytest.mark.parametrize("eb", [1, 2])
def test_repack_build_layout_cases(dev, ref, counts, eb):
    """The digest's _build_layout cases: empty experts, one hot expert, counts
    at / over capacity; distinct per-row values with alternating column gain."""
    H, align, cap, L = 64, 4, 8, len(counts)
    psum, starts, R = build_layout(counts, align)
    base = np.zeros((R, H), np.float32)
    gain = 1.0 + (np.arange(H) % 2)
    for s0, cnt in zip(starts, counts):
        for j in range(cnt):
            base[s0 + j] = float((s0 + j) % 200 + 1) * gain
    if eb == 2:
        exp = synth.to_bf16_bits(base).view(np.uint8).reshape(R, 2 * H)
    else:
        exp = synth.to_e4m3_bits(np.minimum(base, 448)).reshape(R, H)
    st, _, _ = repack_both(dev, ref, exp, eb, H, psum, L, align, cap)
    assert bool(st & ref.ST_OVERFLOW) == any(cnt > cap for cnt in counts)


@pytest.mark.parametrize("fmt", ["packed", "u8", "f32pow2", "f32"])
def test_repack_config_fp8_with_quantizer_scales(dev, ref, fmt):
    """Requant/repack config: 64 experts, 128-aligned psum over 4096 expanded
    rows, e4m3 payload and scales made by each side's own quantiser."""
    d = synth.requant(0)
    c = d["cfg"]
    rng = d["rng"]
    L, align, H, g = c["L"], c["align"], c["H"], 128
    counts = synth.repack_counts(rng, L, c["blocks"], align)
    psum, starts, R = build_layout(counts, align)
    assert R == c["T"]
    cap = int(-(-counts.max() // 128) * 128)
    x = synth.normal_bf16(rng, (R, H))
    G = H // g
    exp = np.zeros((R, H), np.uint8)
    esc, ld_es = ref.scale_buffer(fmt, R, G, fill=0)
    ref.quant_group(x, R, R, H, g, fmt, exp, esc, ld_es)
    # the GPU quantiser must produce the same bytes
    gq = dev.quant_group(bf16_dev(x), group_size=g, scale_fmt=fmt)
    torch.cuda.synchronize()
    assert_same("gpu quantiser payload", to_host(gq["xq"], exp), exp)
    assert_same("gpu quantiser scales", to_host(gq["scales"], esc), esc)
    st, _, _ = repack_both(dev, ref, exp, 1, H, psum, L, align, cap, fmt=fmt, g=g, exp_sc=esc, ld_es=ld_es)
    assert st == 0
    assert cap > 128, "the seeded counts give an expert with more than one block"
    # overflow: capacity one block below the largest expert
    st, _, _ = repack_both(dev, ref, exp, 1, H, psum, L, align, cap - 128, fmt=fmt, g=g, exp_sc=esc, ld_es=ld_es)
    assert st & ref.ST_OVERFLOW


def test_repack_mx_group32_scales(dev, ref):
    """OCP MX (group 32) scales through expanded -> slab -> expanded, H = 224
    (7 groups: not a multiple of 4)."""
    H, g, align, cap = 224, 32, 8, 16
    counts = [5, 0, 16, 3, 9]
    psum, starts, R = build_layout(counts, align)
    rng = np.random.default_rng(31)
    x = synth.normal_bf16(rng, (R, H), outlier_frac=0.05)
    exp = np.zeros((R, H), np.uint8)
    esc, ld_es = ref.scale_buffer("mx", R, H // g, fill=0)
    ref.quant_group(x, R, R, H, g, "mx", exp, esc, ld_es)
    gq = dev.quant_group(bf16_dev(x), group_size=g, scale_fmt="mx")
    torch.cuda.synchronize()
    assert_same("gpu mx payload", to_host(gq["xq"], exp), exp)
    assert_same("gpu mx scales", to_host(gq["scales"], esc), esc)
    repack_both(dev, ref, exp, 1, H, psum, len(counts), align, cap, fmt="mx", g=g, exp_sc=esc, ld_es=ld_es)


def test_repack_weighted_bf16(dev, ref):
    rng = np.random.default_rng(21)
    counts = [5, 0, 130, 1, 77]
    H, align, cap, L = 512, 128, 256, 5
    psum, starts, R = build_layout(counts, align)
    exp = synth.normal_bf16(rng, (R, H)).view(np.uint8).reshape(R, 2 * H)
    wts = rng.random(R).astype(np.float32)
    repack_both(dev, ref, exp, 2, H, psum, L, align, cap, weights=wts)


@pytest.mark.parametrize("eb,H,weighted", [(2, 7184, True), (1, 7184, False), (2, 7168, False)])
def test_repack_multi_segment_rows(dev, ref, eb, H, weighted):
    """Rows longer than one 3.5 KB copy segment, with a ragged last segment
    (H = 7184: 449 or 898 chunks of 16 bytes)."""
    rng = np.random.default_rng(H + eb)
    counts = [3, 0, 140, 1, 30]
    align, cap, L = 128, 256, len(counts)
    psum, starts, R = build_layout(counts, align)
    if eb == 2:
        exp = synth.normal_bf16(rng, (R, H)).view(np.uint8).reshape(R, 2 * H)
    else:
        exp = rng.integers(0, 256, size=(R, H), dtype=np.uint8)
        exp[(exp & 0x7F) == 0x7F] = 0x11          # no NaN codes
    wts = rng.random(R).astype(np.float32) if weighted else None
    repack_both(dev, ref, exp, eb, H, psum, L, align, cap, weights=wts)


def test_repack_bad_layout_flagged(dev, ref):
    H, L, align, cap = 16, 3, 4, 8
    exp = np.zeros((12, H), np.uint8)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    slab = torch.zeros((L * cap, H), dtype=torch.uint8, device=DEV)
    mm = torch.zeros(L, dtype=torch.int32, device=DEV)
    for psum in ([3, 2, 9], [3, 6, 20]):   # a negative count; an end past the buffer (+ overflow)
        st.zero_()
        assert dev.moe_expand_to_slab(to_dev(exp), 1, H, 12, None, 0, to_dev(np.array(psum, np.int32)),
                                      L, align, cap, "u8", 128, slab, None, 0, mm, st) == 0
        assert dev.moe_status_sync(st) == dev.MOE_ERR_BAD_LAYOUT   # the most severe bit wins
        assert int(st.item()) & dev.STATUS_BAD_LAYOUT


def test_binding_allocating_wrappers_repack_and_requant(dev, ref):
    """The allocating wrappers of the binding: quant_group -> expand_to_slab ->
    expand_from_slab round trip (e4m3 rows with packed scales, and weighted
    bf16 rows) against the oracle, and requant in each scale format / mode."""
    rng = np.random.default_rng(77)
    counts = [3, 0, 140, 1, 30]
    H, g, align, cap, L = 1024, 128, 128, 256, len(counts)
    psum, starts, R = build_layout(counts, align)
    x = synth.normal_bf16(rng, (R, H), outlier_frac=0.02)
    q = dev.quant_group(bf16_dev(x), group_size=g, scale_fmt="packed")
    fwd = dev.expand_to_slab(q["xq"], to_dev(psum), L, cap, align=align, exp_scales=q["scales"],
                             ld_es=q["ld_s"], scale_fmt="packed", group_size=g)
    back = dev.expand_from_slab(fwd["slab"], to_dev(psum), R, align=align,
                                slab_scales=fwd["scales"], ld_ss=fwd["ld_s"], scale_fmt="packed",
                                group_size=g)
    torch.cuda.synchronize()
    exp = np.zeros((R, H), np.uint8)
    esc, ld_es = ref.scale_buffer("packed", R, H // g, fill=0)
    ref.quant_group(x, R, R, H, g, "packed", exp, esc, ld_es)
    real = np.concatenate([np.arange(s0, s0 + c) for s0, c in zip(starts, counts)])
    assert np.array_equal(back["exp"].cpu().numpy()[real], exp[real])
    assert np.array_equal(fwd["masked_m"].cpu().numpy(), np.minimum(counts, cap))
    mi_want = np.full(R, -1, np.int32)
    for e, (s0, c) in enumerate(zip(starts, counts)):
        mi_want[s0:s0 + c] = e
    assert np.array_equal(back["m_indices"].cpu().numpy(), mi_want)
    got_sc = back["scales"].cpu().numpy().reshape(-1, back["ld_s"])[:, real]
    assert np.array_equal(got_sc, esc.view(np.int32).reshape(-1, ld_es)[:, real])
    # weighted bf16 rows
    yb = synth.normal_bf16(rng, (R, H))
    wts = rng.random(R).astype(np.float32)
    fwd2 = dev.expand_to_slab(bf16_dev(yb), to_dev(psum), L, cap, align=align)
    back2 = dev.expand_from_slab(fwd2["slab"], to_dev(psum), R, align=align, row_weights=to_dev(wts))
    torch.cuda.synchronize()
    want = np.full((R, 2 * H), 0, np.uint8)
    slab = np.full((L * cap, 2 * H), 0, np.uint8)
    mm = np.zeros(L, np.int32)
    ref.expand_to_slab(yb.view(np.uint8).reshape(R, 2 * H), 2, H, R, None, 0, psum, L, align, cap,
                       "u8", g, slab, None, 0, mm)
    mi = np.zeros(R, np.int32)
    ref.expand_from_slab(slab, 2, H, None, 0, psum, L, align, cap, "u8", g, wts, want, R, None, 0, mi)
    got = back2["exp"].view(torch.int16).cpu().numpy().view(np.uint8).reshape(R, 2 * H)
    assert np.array_equal(got[real], want[real])
    # requant, every scale format and mode
    dq = synth.requant(9, T=64, H=H)
    s8 = np.random.default_rng(5).integers(100, 150, size=64).astype(np.uint8)
    for s_fmt, s_tok in (("f32", dq["s_tok"]), ("ue8m0", s8)):
        for mode in ("max_scale", "amax"):
            qo, S = dev.requant(to_dev(dq["q"]), to_dev(s_tok), s_fmt=s_fmt, mode=mode)
            torch.cuda.synchronize()
            want_q, want_S = ref.requant_ex(dq["q"], s_tok, 64, H, s_fmt, mode)
            assert np.array_equal(qo.cpu().numpy(), want_q), (s_fmt, mode)
            assert float(S.item()) == want_S


# ---------------------------------------------------------------------------
# requant
# ---------------------------------------------------------------------------

def requant_both(dev, ref, q, s):
    T, H = q.shape
    want, S = ref.requant(q, s, T, H)
    out = torch.full((T, H), 0xEE, dtype=torch.uint8, device=DEV)
    dS = torch.zeros(1, dtype=torch.float32, device=DEV)
    assert dev.fp8_requant_per_tensor(to_dev(q), H, to_dev(s), T, H, out, dS) == 0
    torch.cuda.synchronize()
    assert_same("requant payload", to_host(out, want), want)
    assert float(dS.item()) == S


def test_requant_config_full(dev, ref):
    d = synth.requant(0)
    requant_both(dev, ref, d["q"], d["s_tok"])


@pytest.mark.parametrize("T,H", [(1, 16), (37, 1040), (300, 7168), (5, 7184), (33, 3600), (3, 32768)])
def test_requant_shapes(dev, ref, T, H):
    """Rows of one, several and a ragged last segment of the conversion
    launch's 3.5 KB segments."""
    d = synth.requant(T, T=T, H=H)
    requant_both(dev, ref, d["q"], d["s_tok"])


def test_requant_edge_cases(dev, ref):
    q = np.array([[0x38, 0xC0, 0x00, 0x7E] * 4, [0x38, 0x44, 0x80, 0x7E] * 4], np.uint8)
    requant_both(dev, ref, q, np.array([2.0, 1.0], np.float32))
    requant_both(dev, ref, q, np.zeros(2, np.float32))
    dS = torch.zeros(1, dtype=torch.float32, device=DEV)
    assert dev.fp8_requant_per_tensor(None, 16, None, 0, 16, None, dS) == 0
    torch.cuda.synchronize()
    assert float(dS.item()) == 1.0


@pytest.mark.parametrize("s_fmt,mode", [("f32", "max_scale"), ("f32", "amax"), ("ue8m0", "max_scale"),
                                        ("ue8m0", "amax")])
@pytest.mark.parametrize("T,H", [(4096, 7168), (37, 1040)])
def test_requant_ex(dev, ref, s_fmt, mode, T, H):
    d = synth.requant(7, T=T, H=H)
    q = d["q"]
    if s_fmt == "f32":
        s = d["s_tok"]
    else:
        s = np.random.default_rng(T).integers(100, 150, size=T).astype(np.uint8)
    want, S = ref.requant_ex(q, s, T, H, s_fmt, mode)
    out = torch.full((T, H), 0xEE, dtype=torch.uint8, device=DEV)
    dS = torch.zeros(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(T, dtype=torch.float32, device=DEV)
    assert dev.fp8_requant_per_tensor_ex(to_dev(q), H, to_dev(s), s_fmt, T, H, mode, out, dS, ws,
                                         ws.numel() * 4) == 0
    torch.cuda.synchronize()
    assert_same("requant_ex payload", to_host(out, want), want)
    assert float(dS.item()) == S


# ---------------------------------------------------------------------------
# CUDA graph capture and replay
# ---------------------------------------------------------------------------

def test_graph_capture_replay_new_routing(dev, ref):
    T, H, K, E, L, b, g = 256, 1024, 8, 64, 64, 128, 128
    d0 = synth.prefill(0, T=T, H=H)
    ids0 = np.ascontiguousarray(d0["topk_ids"] % E).astype(np.int32)
    x = bf16_dev(d0["x"])
    ids = to_dev(ids0)
    w = to_dev(d0["topk_weights"])
    bound = dev.moe_compact_bound(T * K, L, b)
    rng = np.random.default_rng(3)
    y = bf16_dev(synth.normal_bf16(rng, (bound, H)))
    ws = dev.Workspace(T, K, L, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = dev.dispatch_compact(x, ids, w, E, L, block_e=b, group_size=g, scale_fmt="packed",
                                   workspace=ws, status=st)
        comb = dev.combine(y, out["src2dst"], w, status=st)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = dev.dispatch_compact(x, ids, w, E, L, block_e=b, group_size=g, scale_fmt="packed",
                                   workspace=ws, status=st)
        comb = dev.combine(y, out["src2dst"], w, status=st, out=comb)
    for seed in (1, 2):
        dn = synth.prefill(seed, T=T, H=H)
        idn = np.ascontiguousarray(dn["topk_ids"] % E).astype(np.int32)
        x.copy_(bf16_dev(dn["x"]))
        ids.copy_(to_dev(idn))
        w.copy_(to_dev(dn["topk_weights"]))
        graph.replay()
        torch.cuda.synchronize()
        rxq = np.zeros((bound, H), np.uint8)
        rsc, ld = ref.scale_buffer("packed", bound, H // g)
        rmi = np.zeros(bound, np.int32)
        rs2d = np.zeros((T, K), np.int32)
        rc, rs, rp = (np.zeros(L, np.int32) for _ in range(3))
        rt = np.zeros(1, np.int32)
        ref.dispatch_compact(dn["x"], T, T, H, idn, dn["topk_weights"], K, L, b, g, "packed", rxq,
                             rsc, ld, rmi, bound, rs2d, rc, rs, rp, rt)
        assert np.array_equal(out["src2dst"].cpu().numpy(), rs2d)
        assert np.array_equal(out["m_indices"].cpu().numpy(), rmi)
        rows = rs2d[rs2d >= 0]
        assert np.array_equal(out["xq"].cpu().numpy()[rows], rxq[rows])
        ynp = to_host(y.view(torch.int16), np.zeros((bound, H), np.uint16))
        want = ref.combine_f32(ynp, rs2d, dn["topk_weights"], T, K, H)
        assert_same("graph combine", to_host(comb.view(torch.int16), want), want)
    assert int(st.item()) == 0


def test_graph_capture_replay_with_counter_tail(dev, ref):
    """The dispatch captured once at a size where the staged scatter takes
    its last tokens from the counter (8192 tokens, H = 5248, every expert
    local), then replayed on new routing: the route plan inside the graph
    resets the counter on every replay, and every output buffer (padding rows
    pre-filled with sentinels) matches the oracle."""
    T, H, K, E, L, b, g = 8192, 5248, 8, 256, 256, 128, 128
    G = H // g
    bound = ref.compact_bound(T * K, L, b)
    sent = {"xq": np.full((bound, H), 0xEE, np.uint8)}
    sent["sc"], ld = ref.scale_buffer("packed", bound, G, fill=0xA5)
    sent["mi"] = np.full(bound, -7, np.int32)
    sent["s2d"] = np.full((T, K), -9, np.int32)
    for k in ("counts", "starts", "psum"):
        sent[k] = np.full(L, -5, np.int32)
    sent["total"] = np.full(1, -3, np.int32)
    sent["rw"] = np.full(bound, np.nan, np.float32)
    d = {k: to_dev(v.copy()) for k, v in sent.items()}
    rng = np.random.default_rng(71)
    x = bf16_dev(synth.normal_bf16(rng, (T, H)))
    ids = to_dev(synth.uniform_topk(rng, T, E, K))
    w = to_dev(synth.softmax_weights(rng, T, K))
    ws = dev.Workspace(T, K, L, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)

    def call():
        assert dev.moe_dispatch_compact(x, H, T, None, H, ids, w, K, E, L, b, g, "packed", d["xq"],
                                        d["sc"], ld, d["mi"], bound, d["s2d"], d["counts"],
                                        d["starts"], d["psum"], d["total"], d["rw"], ws.buf,
                                        ws.nbytes, st) == dev.MOE_OK
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for seed in (1, 2):
        rn = np.random.default_rng(71 + seed)
        xh = synth.normal_bf16(rn, (T, H))
        idh = synth.uniform_topk(rn, T, E, K)
        wh = synth.softmax_weights(rn, T, K)
        x.copy_(bf16_dev(xh))
        ids.copy_(to_dev(idh))
        w.copy_(to_dev(wh))
        for k, v in sent.items():
            d[k].copy_(to_dev(v))
        graph.replay()
        torch.cuda.synchronize()
        r = {k: v.copy() for k, v in sent.items()}
        st_ref = ref.dispatch_compact(xh, T, T, H, idh, wh, K, L, b, g, "packed", r["xq"], r["sc"],
                                      ld, r["mi"], bound, r["s2d"], r["counts"], r["starts"],
                                      r["psum"], r["total"], r["rw"])
        assert st_ref == 0
        for k, v in r.items():
            assert_same(f"replay {seed}: {k}", to_host(d[k], v), v)
    assert int(st.item()) == 0


def test_graph_capture_scatter_above_48k_shared_memory(dev, ref):
    """Capture of a two-launch dispatch whose scatter CTA needs more than the
    default 48 KiB of shared memory (1024 experts, 15 chunks: a 60 KiB chunk
    table, staged path since K*L/E = 4), so the launch opts in while the stream
    is being captured; replays with new routing must match the oracle."""
    T, H, K, E, L, b, g = 900, 4096, 4, 1024, 1024, 16, 128
    rng = np.random.default_rng(41)
    x = bf16_dev(synth.normal_bf16(rng, (T, H)))
    ids = to_dev(synth.uniform_topk(rng, T, E, K))
    w = to_dev(synth.softmax_weights(rng, T, K))
    ws = dev.Workspace(T, K, L, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = dev.dispatch_compact(x, ids, w, E, L, block_e=b, group_size=g, scale_fmt="u8",
                                   workspace=ws, status=st)
    bound = dev.moe_compact_bound(T * K, L, b)
    for seed in (5, 6):
        r = np.random.default_rng(seed)
        xn = synth.normal_bf16(r, (T, H))
        idn = synth.uniform_topk(r, T, E, K)
        wn = synth.softmax_weights(r, T, K)
        x.copy_(bf16_dev(xn))
        ids.copy_(to_dev(idn))
        w.copy_(to_dev(wn))
        graph.replay()
        torch.cuda.synchronize()
        rxq = np.zeros((bound, H), np.uint8)
        rsc, ld = ref.scale_buffer("u8", bound, H // g)
        rmi = np.zeros(bound, np.int32)
        rs2d = np.zeros((T, K), np.int32)
        rc, rs, rp = (np.zeros(L, np.int32) for _ in range(3))
        rt = np.zeros(1, np.int32)
        ref.dispatch_compact(xn, T, T, H, idn, wn, K, L, b, g, "u8", rxq, rsc, ld, rmi, bound, rs2d,
                             rc, rs, rp, rt)
        assert np.array_equal(out["src2dst"].cpu().numpy(), rs2d)
        assert np.array_equal(out["m_indices"].cpu().numpy(), rmi)
        rows = rs2d[rs2d >= 0]
        assert np.array_equal(out["xq"].cpu().numpy()[rows], rxq[rows])
        assert np.array_equal(out["scales"].cpu().numpy()[rows], rsc[rows])
    assert int(st.item()) == 0


# ---------------------------------------------------------------------------
# Maximum sizes
# ---------------------------------------------------------------------------

def test_dispatch_max_assignments(dev, ref):
    """T*K = 2^20 slots (the largest accepted) over 256 experts: 64 route-plan
    chunks of 16384 slots (32 warps x 16 steps), a full 64 KiB chunk table."""
    rng = np.random.default_rng(20)
    T, K, L, H = 131072, 8, 256, 128
    x = synth.normal_bf16(rng, (T, H))
    ids = rng.integers(-1, L + 2, size=(T, K)).astype(np.int32)   # a few dropped slots
    w = rng.random((T, K)).astype(np.float32)
    assert dev.moe_workspace_bytes(T, K, L) == 256 + 16384 * 4
    compact_both(dev, ref, x, ids, w, H, K, L + 2, L, 128, 128, "packed", with_rw=False)


# Each case selects one route-plan chain length (slots per lane S) at 32 warps
# per CTA, with the small-table preference of narrow rows (<= 2048 entries):
# 3000 slots x 16 experts: S = 1 (3 chunks); then 64 experts at 40000 / 100000 /
# 200000 / 400000 slots: S = 2 / 4 / 8 / 16 (20 to 25 chunks).
@pytest.mark.parametrize("n_live", [None, 1777, 100, 0])
def test_dispatch_direct_token_counter(dev, ref, n_live):
    """Few kept slots per token (32 of 256 experts local, top-8) with rows of
    two chunks per scatter thread: the scatter takes its tokens from the
    counter that the route plan resets, with a device live count below the
    token count (and below the grid: 100, and 0), compact and masked."""
    rng = np.random.default_rng(31 + (n_live or 0))
    T, K, E, L, H = 3000, 8, 256, 32, 7168
    x = synth.normal_bf16(rng, (T, H), outlier_frac=0.01)
    ids = synth.uniform_topk(rng, T, E, K)
    w = synth.softmax_weights(rng, T, K)
    compact_both(dev, ref, x, ids, w, H, K, E, L, 128, 128, "packed", n_live=n_live)
    masked_both(dev, ref, x, ids, w, H, K, E, L, 128, 128, "packed", n_live=n_live)
    compact_both(dev, ref, x, ids, w, H, K, E, L, 128, 32, "mx", n_live=n_live)


@pytest.mark.parametrize("case", ["all_local", "live_count", "remote_tokens", "overflow", "top6",
                                  "narrow_masked"])
def test_dispatch_staged_tail_from_counter(dev, ref, case):
    """Rows of two chunks per scatter thread (H = 5248) and 8192 tokens: with
    at most 4 scatter CTAs per SM on 152 SMs every CTA has at least 13 tokens,
    so the staged scatter takes its last tokens' worth from the counter that
    the route plan resets. Cases: every expert local (the deep tail), compact
    and masked; a device live count that ends inside the counter's range;
    192 of 256 experts local (6 kept slots per token expected: a one-token
    tail) with a quarter of the tokens routed only to remote experts (claimed
    tokens with no kept slot are skipped), compact and masked; a masked
    capacity below the busiest experts' counts (rows past it dropped, the
    overflow flag set) with the deep tail; top-6 of 160 local experts (the
    count-scaled tail); and rows of one chunk per thread (H = 2048, 16384
    tokens, top-6 of 64: the one-token tail), masked, with a device live
    count."""
    rng = np.random.default_rng(57 + len(case))
    T, K, E, H = 8192, 8, 256, 5248
    x = synth.normal_bf16(rng, (T, H), outlier_frac=0.01)
    ids = synth.uniform_topk(rng, T, E, K)
    w = synth.softmax_weights(rng, T, K)
    if case == "all_local":
        compact_both(dev, ref, x, ids, w, H, K, E, E, 128, 128, "packed")
        masked_both(dev, ref, x, ids, w, H, K, E, E, 384, 128, "packed")
    elif case == "live_count":
        compact_both(dev, ref, x, ids, w, H, K, E, E, 128, 128, "packed", n_live=7900)
    elif case == "overflow":
        masked_both(dev, ref, x, ids, w, H, K, E, E, 256, 128, "packed")
    elif case == "narrow_masked":
        Tn, Hn, Kn, En = 16384, 2048, 6, 64
        xn = synth.normal_bf16(rng, (Tn, Hn))
        idn = synth.uniform_topk(rng, Tn, En, Kn)
        wn = synth.softmax_weights(rng, Tn, Kn)
        masked_both(dev, ref, xn, idn, wn, Hn, Kn, En, En, 2048, 128, "packed", n_live=16000)
    elif case == "top6":
        K6, E6 = 6, 160
        ids6 = synth.uniform_topk(rng, T, E6, K6)
        w6 = synth.softmax_weights(rng, T, K6)
        compact_both(dev, ref, x, ids6, w6, H, K6, E6, E6, 128, 128, "packed")
    else:
        L = 192
        remote = rng.random(T) < 0.25
        ids[remote] = L + synth.uniform_topk(rng, int(remote.sum()), E - L, K)
        compact_both(dev, ref, x, ids, w, H, K, E, L, 128, 128, "packed")
        masked_both(dev, ref, x, ids, w, H, K, E, L, 384, 128, "u8")


@pytest.mark.parametrize("T,L", [(375, 16), (5000, 64), (12500, 64), (25000, 64), (50000, 64)])
def test_dispatch_route_chain_lengths(dev, ref, T, L):
    rng = np.random.default_rng(T + L)
    K, H = 8, 128
    x = synth.normal_bf16(rng, (T, H))
    ids = synth.zipf_topk(rng, T, L, K, n_empty=2)
    w = synth.softmax_weights(rng, T, K)
    compact_both(dev, ref, x, ids, w, H, K, L, L, 128, 128, "packed")


def test_dispatch_long_route_chain(dev, ref):
    """1024 local experts x 262144 slots: only 8 warps fit the per-warp
    histograms, so each lane walks 64 slots (16 chunks of 16384, a full
    64 KiB table)."""
    rng = np.random.default_rng(23)
    T, K, L, H = 8192, 32, 1024, 128
    x = synth.normal_bf16(rng, (T, H))
    ids = synth.zipf_topk(rng, T, L, K, n_empty=24)
    w = synth.softmax_weights(rng, T, K)
    assert dev.moe_workspace_bytes(T, K, L) == 256 + 16384 * 4
    compact_both(dev, ref, x, ids, w, H, K, L, L, 128, 128, "packed")
    masked_both(dev, ref, x, ids, w, H, K, L, L, 256, 128, "packed")


# one launch; two launches: direct (K*L/E = 2), staged (4), staged with the counter tail (8)
@pytest.mark.parametrize("T,K", [(9, 2), (1100, 2), (1100, 4), (2000, 8)])
def test_dispatch_max_hidden(dev, ref, T, K):
    """H = 32768: the two-launch scatter covers the row with 1024 threads x 2
    chunks of 16 in one pass (staged: four 32 KiB staging buffers); the
    one-launch path loops four passes. With 2000 tokens and every slot kept, a
    CTA per SM has 13 tokens and takes the last ones from the counter."""
    rng = np.random.default_rng(21 + K)
    L, H = 8, 32768
    x = synth.normal_bf16(rng, (T, H), outlier_frac=0.01)
    ids = synth.uniform_topk(rng, T, L, K)
    w = synth.softmax_weights(rng, T, K)
    compact_both(dev, ref, x, ids, w, H, K, L, L, 128, 128, "packed")
    masked_both(dev, ref, x, ids, w, H, K, 16, L, 8, 128, "u8")


@pytest.mark.parametrize("H,g,fmt", [(5120, 128, "packed"), (5248, 128, "packed"),
                                     (5120, 32, "mx"), (5152, 32, "u8")])
def test_scatter_chunks_per_thread_boundary(dev, ref, H, g, fmt):
    """Rows of at most 5120 elements run the scatter with one 16-element chunk
    per thread (320 threads at 5120), wider ones with two (5248: 164 threads
    rounded up to 192, the last warp partly idle). Compact (staged, K*L/E = 4),
    masked with direct stores (K*L/E = 1) and the live-row quantiser."""
    rng = np.random.default_rng(H + g)
    T, K = 700, 4
    x = synth.normal_bf16(rng, (T, H), outlier_frac=0.01)
    ids = synth.zipf_topk(rng, T, 64, K, n_empty=4)
    w = synth.softmax_weights(rng, T, K)
    compact_both(dev, ref, x, ids, w, H, K, 64, 64, 128, g, fmt)
    masked_both(dev, ref, x, ids, w, H, K, 64, 16, 256, g, fmt)
    G = H // g
    rxq = np.full((T, H), 0xEE, np.uint8)
    rsc, ld = ref.scale_buffer(fmt, T, G, fill=0x5A)
    ref.quant_group(x, T, 613, H, g, fmt, rxq, rsc, ld)
    dxq, dsc = to_dev(rxq.copy()), to_dev(rsc.copy())
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    nl = torch.tensor([613], dtype=torch.int32, device=DEV)
    assert dev.moe_quant_group(bf16_dev(x), H, T, nl, H, g, fmt, dxq, dsc, ld, st) == 0
    torch.cuda.synchronize()
    assert_same("xq", to_host(dxq, rxq), rxq)
    assert_same("scales", to_host(dsc, rsc), rsc)


@pytest.mark.parametrize("T", [64, 100])     # 2048 slots: one launch; 3200: two launches
def test_dispatch_max_topk_and_experts(dev, ref, T):
    """K = 32 slots per token over L = 1024 local experts."""
    rng = np.random.default_rng(22 + T)
    K, L, H = 32, 1024, 256
    x = synth.normal_bf16(rng, (T, H))
    ids = synth.uniform_topk(rng, T, L, K)
    w = synth.softmax_weights(rng, T, K)
    compact_both(dev, ref, x, ids, w, H, K, L, L, 128, 128, "u8")
    y = synth.normal_bf16(rng, (dev.moe_compact_bound(T * K, L, 128), H))
    r, _, _ = compact_both(dev, ref, x, ids, w, H, K, L, L, 128, 128, "packed")
    check_combine(dev, ref, y, r["s2d"], w, H)


def test_dispatch_max_experts_two_launch(dev, ref):
    """L = 1024 with 160000 slots: 10 chunks x 1024 experts, within the 64 KiB table."""
    rng = np.random.default_rng(23)
    T, K, L, H = 20000, 8, 1024, 128
    x = synth.normal_bf16(rng, (T, H))
    ids = synth.zipf_topk(rng, T, L, K, n_empty=40)
    w = synth.softmax_weights(rng, T, K)
    compact_both(dev, ref, x, ids, w, H, K, L, L, 128, 128, "packed", with_rw=False)
    masked_both(dev, ref, x, ids, w, H, K, L, L, 512, 128, "packed")
