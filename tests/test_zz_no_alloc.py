"""moe_dispatch_compact_noalloc: the compact dispatch for callers that cannot
allocate device memory (graph-capture regions, plugins whose host engine owns
every allocation, serving loops that forbid allocation after start-up). Its
scratch is a static device array inside the library instead of a workspace
the caller allocates.

Checked through the C ABI against moe_dispatch_compact on the same inputs, on
two calls in a row with different routing (the array keeps the first call's
contents, so the second call shows that what must start at zero is cleared).
Dispatch results are integers and bytes, so the comparison is bit-exact.
This file is collected last on purpose.
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
    x = torch.from_numpy(d["x"].view(np.int16)).to(DEV).view(torch.bfloat16)
    return x, torch.from_numpy(ids).to(DEV), torch.from_numpy(d["topk_weights"]).to(DEV)


def _outputs(mp, T, H, K, L, b, g):
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


def test_noalloc_matches_workspace_dispatch_two_calls(dev):
    # 5120 slots: above the 4096-slot one-launch path, so the two-launch path
    # runs and its chunk table lives in the library's static scratch array
    T, H, K, E, L, b, g = 640, 1024, 8, 256, 256, 128, 128
    assert T * K > 4096
    assert dev.moe_workspace_bytes(T, K, L) <= 64 * 1024 + 256
    ws = dev.Workspace(T, K, L, DEV)
    for seed in (0, 1):
        x, ids, w = _inputs(seed, T, H, E)
        ref, bound, ld = _outputs(dev, T, H, K, L, b, g)
        got, _, _ = _outputs(dev, T, H, K, L, b, g)
        a = _args(x, ids, w, T, H, K, E, L, b, g, ref, bound, ld)
        assert dev.moe_dispatch_compact(*a, ws.buf, ws.nbytes, ref["status"]) == dev.MOE_OK
        a = _args(x, ids, w, T, H, K, E, L, b, g, got, bound, ld)
        assert dev.moe_dispatch_compact_noalloc(*a, got["status"]) == dev.MOE_OK
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(ref[k].view(torch.uint8), got[k].view(torch.uint8)), f"call {seed}: {k}"
        assert dev.moe_status_sync(got["status"]) == dev.MOE_OK


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
