"""Host-side checks of the C ABI (no GPU work): the library loads, exports every
symbol include/moeperm.h declares, the host helpers agree with the oracle, and
argument errors are rejected before any launch (pointers here are fake and
never dereferenced)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mp():
    from combine_fp8_quant_gb300 import build
    build.build()
    import combine_fp8_quant_gb300 as m
    m.load()
    return m


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "moeperm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z][a-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(mp):
    names = declared_symbols()
    assert len(names) >= 13
    for n in names:
        assert hasattr(mp.lib(), n), f"missing export {n}"


def test_host_helpers_match_oracle(mp, ref):
    for A, L, b in [(32, 8, 128), (65536, 256, 128), (0, 4, 8), (7, 3, 2), (1000, 7, 16)]:
        assert mp.moe_compact_bound(A, L, b) == ref.compact_bound(A, L, b)
    for E, L in [(256, 32), (256, 33), (8, 8), (64, 16)]:
        assert mp.moe_should_use_masked(E, L) == ref.should_use_masked(E, L)
    for fmt, rows, H, g in [("u8", 112, 7168, 32), ("packed", 98048, 7168, 128), ("f32pow2", 5, 640, 128),
                            ("packed", 13, 640, 128), ("u8", 0, 7168, 32)]:
        assert mp.moe_scale_bytes(fmt, rows, H, g) == ref.scale_bytes(fmt, rows, H, g)
    for fmt, rows, H, g in [("f32", 7, 640, 128), ("mx", 112, 7168, 32)]:
        assert mp.moe_scale_bytes(fmt, rows, H, g) == ref.scale_bytes(fmt, rows, H, g)
    assert mp.moe_scale_bytes("packed", 10, 7168, 32) == 0      # unsupported pairs
    assert mp.moe_scale_bytes("mx", 10, 7168, 128) == 0
    assert mp.moe_scale_bytes("f32", 10, 7168, 32) == 0
    assert mp.moe_workspace_bytes(8192, 8, 256) >= 256 + 16 * 256 * 4


FAKE = 1 << 20          # a 16-byte aligned fake device address, never dereferenced
ODD = FAKE + 4


def compact_args(**over):
    a = dict(x=FAKE, ldx=7168, T=64, d_num_tokens=None, H=7168, topk_ids=FAKE, topk_weights=FAKE,
             K=8, E=256, L=256, block_e=128, g=128, fmt="packed", xq=FAKE, scales=FAKE,
             ld_s=None, m_indices=FAKE, bound=None, src2dst=FAKE, counts=FAKE, starts=FAKE,
             psum=FAKE, total=FAKE, row_weights=None, workspace=FAKE, workspace_bytes=1 << 20,
             d_status=FAKE)
    a.update(over)
    return a


def call_compact(mp, **over):
    a = compact_args(**over)
    bound = mp.moe_compact_bound(a["T"] * a["K"], a["L"], a["block_e"]) if a["bound"] is None else a["bound"]
    ld = ((bound + 3) // 4 * 4) if a["ld_s"] is None else a["ld_s"]
    a["bound"], a["ld_s"] = bound, ld
    order = ["x", "ldx", "T", "d_num_tokens", "H", "topk_ids", "topk_weights", "K", "E", "L",
             "block_e", "g", "fmt", "xq", "scales", "ld_s", "m_indices", "bound", "src2dst",
             "counts", "starts", "psum", "total", "row_weights", "workspace", "workspace_bytes",
             "d_status"]
    return mp.moe_dispatch_compact(*[a[k] for k in order], stream=_NullStream())


class _NullStream:
    cuda_stream = 0


@pytest.mark.parametrize("over", [
    dict(H=7160), dict(H=7168 + 64), dict(g=64), dict(g=32, fmt="packed"), dict(K=0), dict(K=33),
    dict(L=0), dict(L=1025, E=2000), dict(E=100, L=256), dict(block_e=0), dict(x=ODD),
    dict(xq=ODD), dict(scales=None), dict(ldx=7000), dict(ldx=7172), dict(m_indices=None),
    dict(bound=1000), dict(ld_s=33020), dict(ld_s=33026), dict(workspace_bytes=64),
    dict(workspace=None), dict(row_weights=FAKE, topk_weights=None), dict(T=200000),
    dict(T=-1), dict(src2dst=None), dict(topk_ids=None),
])
def test_dispatch_compact_rejects(mp, over):
    assert call_compact(mp, **over) == mp.MOE_ERR_INVALID_ARG


def test_other_calls_reject(mp):
    S = _NullStream()
    E = mp.MOE_ERR_INVALID_ARG
    # masked: bad cap, missing masked_m, packed ld below cap, psum with a zero alignment
    assert mp.moe_dispatch_masked(FAKE, 7168, 8, None, 7168, FAKE, FAKE, 8, 256, 32, 0, 128, "packed",
                                  FAKE, FAKE, 4, FAKE, FAKE, None, None, 128, FAKE, 1 << 20, FAKE,
                                  S) == E
    assert mp.moe_dispatch_masked(FAKE, 7168, 8, None, 7168, FAKE, FAKE, 8, 256, 32, 16, 128, "packed",
                                  FAKE, FAKE, 16, None, FAKE, None, None, 128, FAKE, 1 << 20, FAKE,
                                  S) == E
    assert mp.moe_dispatch_masked(FAKE, 7168, 8, None, 7168, FAKE, FAKE, 8, 256, 32, 16, 128, "packed",
                                  FAKE, FAKE, 12, FAKE, FAKE, None, None, 128, FAKE, 1 << 20, FAKE,
                                  S) == E
    assert mp.moe_dispatch_masked(FAKE, 7168, 8, None, 7168, FAKE, FAKE, 8, 256, 32, 16, 128, "packed",
                                  FAKE, FAKE, 16, FAKE, FAKE, None, FAKE, 0, FAKE, 1 << 20, FAKE,
                                  S) == E
    # quant_group: packed with g = 32, odd pointer
    assert mp.moe_quant_group(FAKE, 7168, 112, None, 7168, 32, "packed", FAKE, FAKE, 112, FAKE, S) == E
    assert mp.moe_quant_group(ODD, 7168, 112, None, 7168, 32, "u8", FAKE, FAKE, 224, FAKE, S) == E
    # combine: K too large, H not a multiple of 8, unaligned out
    assert mp.moe_combine(FAKE, 7168, 100, FAKE, None, 8, None, 40, 7168, FAKE, FAKE, S) == E
    assert mp.moe_combine(FAKE, 7168, 100, FAKE, None, 8, None, 8, 7164, FAKE, FAKE, S) == E
    assert mp.moe_combine(FAKE, 7168, 100, FAKE, None, 8, None, 8, 7168, ODD, FAKE, S) == E
    # repack: weights on fp8, one scale pointer only, bad elem size
    assert mp.moe_expand_from_slab(FAKE, 1, 7168, None, 0, FAKE, 4, 128, 256, "u8", 128, FAKE,
                                   FAKE, 1024, None, 0, None, FAKE, S) == E
    assert mp.moe_expand_to_slab(FAKE, 1, 7168, 1024, FAKE, 56, FAKE, 4, 128, 256, "u8", 128,
                                 FAKE, None, 56, FAKE, FAKE, S) == E
    assert mp.moe_expand_to_slab(FAKE, 4, 7168, 1024, None, 0, FAKE, 4, 128, 256, "u8", 128,
                                 FAKE, None, 0, FAKE, FAKE, S) == E
    # requant: missing scale output, bad ldq
    assert mp.fp8_requant_per_tensor(FAKE, 7168, FAKE, 16, 7168, FAKE, None, S) == E
    assert mp.fp8_requant_per_tensor(FAKE, 7000, FAKE, 16, 7168, FAKE, FAKE, S) == E
    assert mp.moe_status_sync(None, S) == E
    assert "invalid" in mp.lib().moe_status_string(E).decode()


def test_binding_rejects_cpu_tensors(mp):
    import torch
    x = torch.zeros(16, dtype=torch.uint8)
    with pytest.raises(ValueError):
        mp.moe_quant_group(x, 16, 1, None, 16, 32, "u8", FAKE, FAKE, 1, FAKE, _NullStream())


def test_size_limits_rejected(mp):
    assert call_compact(mp, H=32768 + 128, ldx=32768 + 128) == mp.MOE_ERR_INVALID_ARG
    assert call_compact(mp, T=(1 << 20) // 8 + 1) == mp.MOE_ERR_INVALID_ARG
    # chunk table beyond 64 KiB: 1024 experts with 2^19 slots
    assert mp.moe_workspace_bytes(65536, 8, 1024) == 0
    assert call_compact(mp, T=65536, L=1024, E=1024, workspace_bytes=1 << 24) == mp.MOE_ERR_INVALID_ARG


def _route_geometry_table(A, L, pref):
    """The route-plan geometry rule restated: the shortest chain S (slots per
    lane) in 1, 2, 4, 8, 16 at up to 32 warps (fewer when warps x L would pass
    12288 histogram entries), or 64 at up to 8 warps, whose table (chunks x L)
    fits `pref` entries, else the shortest whose table fits 16384."""
    wmax = 1 if L >= 12288 else min(32, 12288 // L)
    for limit in (pref, 16384):
        for S in (1, 2, 4, 8, 16, 64):
            W = min(wmax, 8 if S > 16 else 32)
            chunk = 32 * W * S
            nc = max(1, -(-A // chunk))
            if nc * L <= limit:
                return nc * L
    return None


@pytest.mark.parametrize("T,K,L", [(300, 8, 256), (8192, 8, 256), (8192, 8, 128), (8192, 8, 32),
                                   (16384, 6, 64), (32768, 8, 256), (131072, 8, 256), (8192, 32, 1024),
                                   (1000, 3, 1), (4096, 8, 160), (50000, 8, 64), (9999, 7, 333)])
def test_workspace_bytes_follow_the_route_geometry(mp, T, K, L):
    """One workspace serves every row width: it holds the larger chunk table of
    the two table preferences (2048 entries for narrow rows or <= 128 local
    experts, 8192 otherwise)."""
    want = max(_route_geometry_table(T * K, L, 2048), _route_geometry_table(T * K, L, 8192))
    assert mp.moe_workspace_bytes(T, K, L) == 256 + 4 * want
