"""The workloads end to end on the GPU, each call compared with the CPU oracle
over whole buffers (sentinel-filled on both sides, so rows the definition does
not name must stay untouched):

  * tiny: compact dispatch, then the weighted combine of N(0,1) expert outputs
    over the 1024-row static bound, on five seeds and every group-128 format;
  * decode (masked): T = 128, hidden 7168, 32 of 256 experts local, top-8,
    slab capacity 128, packed UE8M0 -- the dispatch with its device-side psum
    (PR #29525 实现拆解 item 3, _build_layout), slab -> expanded (psum aligned
    to 128) -> slab (PR #29525 _check_expand_roundtrip), and the weighted
    combine from slab rows; also the variant that applies the weights in
    slab -> expanded on bf16 rows and combines with unit weights; and the
    chain captured once in a CUDA graph, replayed with new routing;
  * prefill (compact): T = 8192, hidden 7168, 256 local experts, top-8 Zipf
    routing, block_e 128, packed UE8M0, in the launch configuration the bench
    times -- every payload byte, every scale word, m_indices, src2dst, counts,
    starts, psum, total, row weights, and all 8192 x 7168 combine outputs;
    the same for two more MoE shapes of the bench's shape sweep.

Layout, payload and scale bytes must be identical; the combine must equal the
oracle's fp32-FMA twin bit for bit and lie within one bf16 ulp of the fp64 sum
plus the fp32 accumulation floor K * 2^-24 * sum |w*y|.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import DEV, bf16_dev, to_dev, to_host
from test_gpu_parity import assert_same, check_combine, compact_both, masked_both

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------------------
# tiny
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("fmt", ["packed", "u8", "f32pow2", "f32"])
def test_tiny_config_end_to_end(dev, ref, seed, fmt):
    d = synth.tiny(seed)
    c = d["cfg"]
    T, H, K, E, L, b, g = c["T"], c["H"], c["K"], c["E"], c["L"], c["block_e"], c["g"]
    r, _, _ = compact_both(dev, ref, d["x"], d["topk_ids"], d["topk_weights"], H, K, E, L, b, g, fmt)
    bound = ref.compact_bound(T * K, L, b)
    assert bound == 1024
    y = synth.expert_outputs(np.random.default_rng(100 + seed), bound, H)
    check_combine(dev, ref, y, r["s2d"], d["topk_weights"], H)


# ---------------------------------------------------------------------------
# decode: masked dispatch -> slab -> expanded -> slab -> weighted combine
# ---------------------------------------------------------------------------

def expanded_starts(psum, align):
    """Segment starts of the expanded layout, align(psum[e-1]) (psum[-1] = 0)."""
    starts, prev = [], 0
    for p in psum:
        starts.append(-(-prev // align) * align)
        prev = int(p)
    return starts


def slab_rows_to_expanded(s2d, psum, cap, align):
    """The expanded row of each slot's slab row e*cap + j: start_e + j."""
    starts = expanded_starts(psum, align)
    out = np.full_like(s2d, -1)
    flat, of = s2d.reshape(-1), out.reshape(-1)
    for a, row in enumerate(flat):
        if row >= 0:
            of[a] = starts[row // cap] + row % cap
    return out


def from_slab_both(dev, ref, slab, d_slab, eb, H, psum, d_psum, L, align, cap, R, fmt=None,
                   ssc=None, d_ssc=None, ld_ss=0, weights=None):
    """slab -> expanded rows on both sides (sentinel-filled outputs), the GPU
    reading the psum the GPU dispatch wrote. Returns the oracle's and the
    GPU's expanded rows (and scales)."""
    G = H // 128
    exp = np.full((R, H * eb), 0xDD, np.uint8)
    mi = np.full(R, 77, np.int32)
    esc, ld_es = (ref.scale_buffer(fmt, R, G, fill=0x11) if ssc is not None else (None, 0))
    st_ref = ref.expand_from_slab(slab, eb, H, ssc, ld_ss, psum, L, align, cap, fmt or "u8", 128,
                                  weights, exp, R, esc, ld_es, mi)
    d_exp, d_mi = to_dev(np.full_like(exp, 0xDD)), to_dev(np.full_like(mi, 77))
    d_esc = to_dev(np.full_like(esc, 0x11)) if esc is not None else None
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert dev.moe_expand_from_slab(d_slab, eb, H, d_ssc, ld_ss, d_psum, L, align, cap, fmt or "u8",
                                    128, to_dev(weights) if weights is not None else None, d_exp, R,
                                    d_esc, ld_es, d_mi, st) == dev.MOE_OK
    torch.cuda.synchronize()
    assert_same("expanded rows", to_host(d_exp, exp), exp)
    assert_same("expanded m_indices", to_host(d_mi, mi), mi)
    if esc is not None:
        assert_same("expanded scales", to_host(d_esc, esc), esc)
    assert int(st.item()) == st_ref == 0
    return dict(exp=exp, esc=esc, ld_es=ld_es, d_exp=d_exp, d_esc=d_esc)


@pytest.mark.parametrize("seed", range(3))
def test_decode_config_chain(dev, ref, seed):
    d = synth.decode(seed)
    c = d["cfg"]
    T, H, K, E, L, cap, g, align = c["T"], c["H"], c["K"], c["E"], c["L"], c["cap"], c["g"], c["align"]
    x, ids, w = d["x"], d["topk_ids"], d["topk_weights"]
    G = H // g

    # 1. masked dispatch (cap 128, packed UE8M0) with its expanded-layout psum
    r, dd, status = masked_both(dev, ref, x, ids, w, H, K, E, L, cap, g, "packed", psum_align=align)
    assert int(status.item()) == 0
    R = ref.compact_bound(T * K, L, align)
    assert r["psum"][-1] <= R

    # 2. slab -> expanded, driven by the device psum
    ssc2, ld_ss = ref.scale_buffer("packed", L * cap, G, fill=0xA5, blocks=L)
    e1 = from_slab_both(dev, ref, r["xq"], dd["xq"], 1, H, r["psum"], dd["psum"], L, align, cap, R,
                        fmt="packed", ssc=r["sc"], d_ssc=dd["sc"], ld_ss=ld_ss)

    # 3. expanded -> slab again: the original slab on real rows, padding untouched
    slab2 = np.full_like(r["xq"], 0xEE)
    mm2 = np.full(L, -1, np.int32)
    st_ref = ref.expand_to_slab(e1["exp"], 1, H, R, e1["esc"], e1["ld_es"], r["psum"], L, align, cap,
                                "packed", g, slab2, ssc2, ld_ss, mm2)
    assert st_ref == 0
    assert np.array_equal(slab2, r["xq"]), "roundtrip returns the dispatched slab"
    assert np.array_equal(ssc2, r["sc"]), "and its scales"
    assert np.array_equal(mm2, r["mm"])
    d_slab2, d_ssc2 = to_dev(np.full_like(slab2, 0xEE)), to_dev(np.full_like(ssc2, 0xA5))
    d_mm2 = to_dev(np.full(L, -1, np.int32))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert dev.moe_expand_to_slab(e1["d_exp"], 1, H, R, e1["d_esc"], e1["ld_es"], dd["psum"], L, align,
                                  cap, "packed", g, d_slab2, d_ssc2, ld_ss, d_mm2, st) == dev.MOE_OK
    torch.cuda.synchronize()
    assert_same("slab after roundtrip", to_host(d_slab2, slab2), slab2)
    assert_same("slab scales after roundtrip", to_host(d_ssc2, ssc2), ssc2)
    assert_same("masked_m after roundtrip", to_host(d_mm2, mm2), mm2)
    assert int(st.item()) == 0

    # 4. weighted combine of bf16 expert outputs read straight from slab rows
    y = synth.expert_outputs(np.random.default_rng(200 + seed), L * cap, H)
    check_combine(dev, ref, y, r["s2d"], w, H)

    # 5. the other reading: weights applied on real rows in slab -> expanded
    #    (bf16), then a unit-weight combine over the expanded rows
    s2d_exp = slab_rows_to_expanded(r["s2d"], r["psum"], cap, align)
    w_exp = np.zeros(R, np.float32)
    w_exp[s2d_exp[s2d_exp >= 0]] = w[s2d_exp >= 0]
    y_slab = y.view(np.uint8).reshape(L * cap, 2 * H)
    e2 = from_slab_both(dev, ref, y_slab, to_dev(y_slab), 2, H, r["psum"], dd["psum"], L, align, cap,
                        R, weights=w_exp)
    y_exp = e2["exp"].view(np.uint16).reshape(R, H)
    check_combine(dev, ref, y_exp, s2d_exp, None, H)


def test_decode_chain_graph_replay_new_routing(dev, ref):
    """The decode chain (masked dispatch with psum, slab -> expanded, expanded
    -> slab, weighted combine) captured once in a CUDA graph and replayed on a
    second routing written into the same input buffers."""
    c = synth.DECODE
    T, H, K, E, L, cap, g, align = c["T"], c["H"], c["K"], c["E"], c["L"], c["cap"], c["g"], c["align"]
    G = H // g
    R = dev.moe_compact_bound(T * K, L, align)
    x, ids, w = (torch.empty((T, H), dtype=torch.bfloat16, device=DEV),
                 torch.empty((T, K), dtype=torch.int32, device=DEV),
                 torch.empty((T, K), dtype=torch.float32, device=DEV))
    y = torch.empty((L * cap, H), dtype=torch.bfloat16, device=DEV)
    xq = torch.empty((L * cap, H), dtype=torch.uint8, device=DEV)
    sc, ld = dev.scale_tensor("packed", L * cap, H, g, DEV, blocks=L)
    mm, psum = torch.empty(L, dtype=torch.int32, device=DEV), torch.empty(L, dtype=torch.int32, device=DEV)
    s2d = torch.empty((T, K), dtype=torch.int32, device=DEV)
    exp = torch.empty((R, H), dtype=torch.uint8, device=DEV)
    esc, ld_es = dev.scale_tensor("packed", R, H, g, DEV)
    mi = torch.empty(R, dtype=torch.int32, device=DEV)
    slab2 = torch.empty_like(xq)
    sc2 = torch.empty_like(sc)
    mm2 = torch.empty_like(mm)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    ws = dev.Workspace(T, K, L, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)

    def chain():
        assert dev.moe_dispatch_masked(x, H, T, None, H, ids, w, K, E, L, cap, g, "packed", xq, sc, ld,
                                       mm, s2d, None, psum, align, ws.buf, ws.nbytes, st) == 0
        assert dev.moe_expand_from_slab(xq, 1, H, sc, ld, psum, L, align, cap, "packed", g, None, exp, R,
                                        esc, ld_es, mi, st) == 0
        assert dev.moe_expand_to_slab(exp, 1, H, R, esc, ld_es, psum, L, align, cap, "packed", g, slab2,
                                      sc2, ld, mm2, st) == 0
        assert dev.moe_combine(y, H, L * cap, s2d, w, T, None, K, H, out, st) == 0

    def load(seed):
        d = synth.decode(seed)
        x.copy_(bf16_dev(d["x"]))
        ids.copy_(to_dev(d["topk_ids"]))
        w.copy_(to_dev(d["topk_weights"]))
        y.copy_(bf16_dev(synth.expert_outputs(np.random.default_rng(300 + seed), L * cap, H)))
        return d

    load(10)
    chain()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            chain()
    torch.cuda.current_stream().wait_stream(s)
    for seed in (11, 12):
        d = load(seed)
        slab2.fill_(0xEE)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert dev.moe_status_sync(st) == dev.MOE_OK
        r = {"xq": np.full((L * cap, H), 0xEE, np.uint8)}
        r["sc"], rld = ref.scale_buffer("packed", L * cap, G, fill=0xA5, blocks=L)
        r["mm"], r["psum"] = np.zeros(L, np.int32), np.zeros(L, np.int32)
        r["s2d"] = np.zeros((T, K), np.int32)
        assert ref.dispatch_masked(d["x"], T, T, H, d["topk_ids"], d["topk_weights"], K, L, cap, g, "packed",
                                   r["xq"], r["sc"], rld, r["mm"], r["s2d"], None, psum=r["psum"],
                                   psum_align=align) == 0
        assert np.array_equal(psum.cpu().numpy(), r["psum"])
        assert np.array_equal(mm2.cpu().numpy(), r["mm"])
        assert np.array_equal(s2d.cpu().numpy(), r["s2d"])
        assert_same("slab after the graph's roundtrip", slab2.cpu().numpy(), r["xq"])
        yh = synth.expert_outputs(np.random.default_rng(300 + seed), L * cap, H)
        want = ref.combine_f32(yh, r["s2d"], d["topk_weights"], T, K, H)
        assert_same("combine", out.view(torch.int16).cpu().numpy().view(np.uint16), want)


# ---------------------------------------------------------------------------
# prefill and the shape sweep: whole buffers at full size
# ---------------------------------------------------------------------------

def whole_buffer_step(dev, ref, x, ids, w, E, L, b=128, g=128, seed=11):
    T, H = x.shape
    K = ids.shape[1]
    r, _, _ = compact_both(dev, ref, x, ids, w, H, K, E, L, b, g, "packed")
    y = synth.expert_outputs(np.random.default_rng(seed), r["xq"].shape[0], H)
    check_combine(dev, ref, y, r["s2d"], w, H)


def test_prefill_config_whole_buffer(dev, ref):
    """T = 8192, H = 7168, 256 local experts, top-8 Zipf routing, block_e 128,
    packed UE8M0: the call the bench times, every output byte against the
    oracle."""
    d = synth.prefill(0)
    c = d["cfg"]
    assert (c["T"], c["H"], c["block_e"], c["g"]) == (8192, 7168, 128, 128)
    whole_buffer_step(dev, ref, d["x"], d["topk_ids"], d["topk_weights"], c["E"], c["L"])


@pytest.mark.parametrize("T,H,E,K", [(16384, 2048, 64, 6), (8192, 5120, 160, 6)])
def test_sweep_shapes_whole_buffer(dev, ref, T, H, E, K):
    """Two shapes of the shape sweep at full size: narrow rows (one chunk per
    scatter thread, the small route-plan table) and top-6 over 160 experts
    (3 + 3 row batches in the combine)."""
    rng = np.random.default_rng(T + H + E + K)
    x = synth.normal_bf16(rng, (T, H))
    ids = synth.zipf_topk(rng, T, E, K, n_empty=12)
    w = synth.softmax_weights(rng, T, K)
    whole_buffer_step(dev, ref, x, ids, w, E, E)
