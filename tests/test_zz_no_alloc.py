"""moe_dispatch_compact_noalloc: the compact dispatch for callers that cannot
allocate device memory -- a plugin whose host engine owns every device
allocation and passes in only inputs and outputs, or a serving loop that
forbids allocation after start-up. Its scratch is a static device array inside
the library instead of a workspace the caller allocates.

Checked through the C ABI, bit for bit (dispatch results are integers and
bytes), against the CPU oracle and against moe_dispatch_compact with a
caller-allocated workspace on the same inputs: on two calls in a row with
different routing (the array keeps the first call's contents, so the second
call shows that nothing it reads is left over from the first), on the
one-launch path (at most 2048 slots, where the scratch is not used) and the
two-launch path (where the chunk table lives in the array), and on an empty
batch. Sizes beyond the array are rejected before any GPU work.

This file is collected last on purpose, and each test sets up its own inputs,
so it passes alone in a fresh process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _inputs(seed, T, H, E):
    d = synth.prefill(seed, T=T, H=H)
    ids = np.ascontiguousarray(d["topk_ids"] % E).astype(np.int32)
    return d["x"], ids, d["topk_weights"]


def _dev_outputs(mp, T, H, K, L, b, g):
    bound = mp.moe_compact_bound(T * K, L, b)
    sc, ld = mp.scale_tensor("packed", bound, H, g, DEV)
    o = dict(xq=torch.full((bound, H), 0xEE, dtype=torch.uint8, device=DEV), sc=sc.fill_(-1),
             mi=torch.full((bound,), -7, dtype=torch.int32, device=DEV),
             s2d=torch.full((T, K), -9, dtype=torch.int32, device=DEV),
             counts=torch.full((L,), -5, dtype=torch.int32, device=DEV),
             starts=torch.full((L,), -5, dtype=torch.int32, device=DEV),
             psum=torch.full((L,), -5, dtype=torch.int32, device=DEV),
             total=torch.full((1,), -3, dtype=torch.int32, device=DEV),
             rw=torch.full((bound,), float("nan"), dtype=torch.float32, device=DEV),
             status=torch.zeros(1, dtype=torch.int32, device=DEV))
    return o, bound, ld


def _args(x, ids, w, T, H, K, E, L, b, g, o, bound, ld):
    return (x, H, T, None, H, ids, w, K, E, L, b, g, "packed", o["xq"], o["sc"], ld, o["mi"], bound,
            o["s2d"], o["counts"], o["starts"], o["psum"], o["total"], o["rw"])


def _oracle(ref, x, ids, w, T, H, K, L, b, g, bound, ld):
    """The oracle on the same sentinels as _dev_outputs (bytes of the packed
    scale buffer start as 0xFF, like the device buffer filled with -1)."""
    r = dict(xq=np.full((bound, H), 0xEE, np.uint8),
             sc=ref.scale_buffer("packed", bound, H // g, fill=0xFF, ld=ld)[0],
             mi=np.full(bound, -7, np.int32), s2d=np.full((T, K), -9, np.int32),
             counts=np.full(L, -5, np.int32), starts=np.full(L, -5, np.int32),
             psum=np.full(L, -5, np.int32), total=np.full(1, -3, np.int32),
             rw=np.full(bound, np.nan, np.float32))
    st = ref.dispatch_compact(x, T, T, H, ids, w, K, L, b, g, "packed", r["xq"], r["sc"], ld, r["mi"],
                              bound, r["s2d"], r["counts"], r["starts"], r["psum"], r["total"], r["rw"])
    return r, st


def _same_bytes(t, a):
    return np.array_equal(t.cpu().numpy().reshape(-1).view(np.uint8),
                          np.ascontiguousarray(a).reshape(-1).view(np.uint8))


@pytest.mark.parametrize("T", [640, 200])   # 5120 slots: two launches; 1600 slots: one launch
def test_noalloc_matches_oracle_and_workspace_dispatch_two_calls(dev, ref, T):
    H, K, E, L, b, g = 1024, 8, 256, 256, 128, 128
    assert (T * K > 2048) == (T == 640)      # the one-launch path takes at most 2048 slots
    assert dev.moe_workspace_bytes(T, K, L) <= 64 * 1024 + 256
    ws = dev.Workspace(T, K, L, DEV)
    for seed in (0, 1):                      # two calls in a row, different routing
        xh, idh, wh = _inputs(seed + T, T, H, E)
        x = torch.from_numpy(xh.view(np.int16)).to(DEV).view(torch.bfloat16)
        ids, w = torch.from_numpy(idh).to(DEV), torch.from_numpy(wh).to(DEV)
        want, bound, ld = _dev_outputs(dev, T, H, K, L, b, g)
        got, _, _ = _dev_outputs(dev, T, H, K, L, b, g)
        a = _args(x, ids, w, T, H, K, E, L, b, g, want, bound, ld)
        assert dev.moe_dispatch_compact(*a, ws.buf, ws.nbytes, want["status"]) == dev.MOE_OK
        a = _args(x, ids, w, T, H, K, E, L, b, g, got, bound, ld)
        assert dev.moe_dispatch_compact_noalloc(*a, got["status"]) == dev.MOE_OK
        torch.cuda.synchronize()
        for k in want:
            assert torch.equal(want[k].view(torch.uint8), got[k].view(torch.uint8)), f"call {seed}: {k}"
        r, st_ref = _oracle(ref, xh, idh, wh, T, H, K, L, b, g, bound, ld)
        assert st_ref == 0 and dev.moe_status_sync(got["status"]) == dev.MOE_OK
        for k in r:
            assert _same_bytes(got[k], r[k]), f"call {seed}: {k} differs from the oracle"


def test_noalloc_empty_batch(dev, ref):
    """T = 0: no rows, every expert empty; the layout outputs are still written."""
    H, K, E, L, b, g = 256, 2, 8, 8, 128, 128
    o = dict(counts=torch.full((L,), -5, dtype=torch.int32, device=DEV),
             starts=torch.full((L,), -5, dtype=torch.int32, device=DEV),
             psum=torch.full((L,), -5, dtype=torch.int32, device=DEV),
             total=torch.full((1,), -3, dtype=torch.int32, device=DEV),
             status=torch.zeros(1, dtype=torch.int32, device=DEV))
    assert dev.moe_compact_bound(0, L, b) == 0
    code = dev.moe_dispatch_compact_noalloc(None, H, 0, None, H, None, None, K, E, L, b, g, "packed",
                                            None, None, 4, None, 0, None, o["counts"], o["starts"],
                                            o["psum"], o["total"], None, o["status"])
    assert code == dev.MOE_OK
    torch.cuda.synchronize()
    r = dict(counts=np.full(L, -5, np.int32), starts=np.full(L, -5, np.int32),
             psum=np.full(L, -5, np.int32), total=np.full(1, -3, np.int32))
    ref.dispatch_compact(np.zeros((0, H), np.uint16), 0, 0, H, np.zeros((0, K), np.int32),
                         np.zeros((0, K), np.float32), K, L, b, g, "packed", np.zeros((0, H), np.uint8),
                         np.zeros(16, np.uint8), 4, np.zeros(0, np.int32), 0, np.zeros((0, K), np.int32),
                         r["counts"], r["starts"], r["psum"], r["total"])
    for k in r:
        assert _same_bytes(o[k], r[k]), k
    assert dev.moe_status_sync(o["status"]) == dev.MOE_OK


def test_noalloc_rejects_sizes_beyond_its_array(dev):
    # 20 chunks x 1024 experts would need an 80 KiB table: beyond the array
    # (and beyond what the dispatch supports at all, so the workspace query says 0)
    T, H, K, L = 40000, 128, 8, 1024
    assert dev.moe_workspace_bytes(T, K, L) == 0
    fake = 1 << 20
    code = dev.moe_dispatch_compact_noalloc(fake, H, T, None, H, fake, None, K, L, L, 128, 128,
                                            "packed", fake, fake, 1 << 20, fake, 1 << 22, fake,
                                            fake, fake, fake, fake, None, fake)
    assert code == dev.MOE_ERR_INVALID_ARG
