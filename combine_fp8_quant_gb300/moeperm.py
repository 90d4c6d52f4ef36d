"""Python binding of libmoeperm (include/moeperm.h).

Thin marshalling only: every function here passes device pointers, sizes and
the current CUDA stream of torch to the C ABI of the same name. All arithmetic
of the path runs in the library's sm_103a kernels; there is no CPU fallback.
If the shared library is missing or cannot be loaded, loading raises.

Two layers:
  * ``moe_*`` / ``fp8_requant_per_tensor``: one-to-one with the C calls, taking
    torch tensors (or None) and returning the status code.
  * ``dispatch_compact`` / ``dispatch_masked`` / ``quant_group`` / ``combine`` /
    ``expand_to_slab`` / ``expand_from_slab`` / ``requant``: allocate the output
    tensors with torch (device memory is PyTorch's job) and call the C ABI.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoeperm.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_OVERFLOW = 0, 1, 2
MOE_ERR_LIVE_OVERFLOW, MOE_ERR_BAD_LAYOUT, MOE_ERR_CUDA = 3, 4, 5
STATUS_OVERFLOW, STATUS_LIVE_OVERFLOW, STATUS_BAD_LAYOUT = 1, 2, 4
FMT = {"u8": 0, "packed": 1, "f32pow2": 2, "f32": 3, "mx": 4}

_lock = threading.Lock()
_lib = None


class MoePermError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = _lib.moe_status_string(code).decode() if _lib is not None else str(code)
        super().__init__(f"{where}: {msg} (status {code})")


def load(path: str | None = None):
    """Load libmoeperm.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libmoeperm.so not found at {p}: build it first (python -c "
                "'import __graft_entry__ as g; g.build()'). There is no CPU fallback.")
        lib = C.CDLL(p)
        _declare(lib)
        _lib = lib
        return lib


def _declare(L):
    vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
    sig = {
        "moe_compact_bound": (i64, [i64, i32, i32]),
        "moe_should_use_masked": (i32, [i32, i32]),
        "moe_scale_bytes": (sz, [i32, i64, i32, i32]),
        "moe_workspace_bytes": (sz, [i32, i32, i32]),
        "moe_dispatch_compact": (i32, [vp, i64, i32, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                       vp, vp, i64, vp, i64, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]),
        "moe_dispatch_masked": (i32, [vp, i64, i32, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                      vp, vp, i64, vp, vp, vp, vp, i32, vp, sz, vp, vp]),
        "moe_dispatch_compact_noalloc": (i32, [vp, i64, i32, vp, i32, vp, vp, i32, i32, i32, i32,
                                               i32, i32, vp, vp, i64, vp, i64, vp, vp, vp, vp, vp,
                                               vp, vp, vp]),
        "moe_quant_group": (i32, [vp, i64, i32, vp, i32, i32, i32, vp, vp, i64, vp, vp]),
        "moe_combine": (i32, [vp, i64, i64, vp, vp, i32, vp, i32, i32, vp, vp, vp]),
        "moe_expand_to_slab": (i32, [vp, i32, i32, i64, vp, i64, vp, i32, i32, i32, i32, i32, vp,
                                     vp, i64, vp, vp, vp]),
        "moe_expand_from_slab": (i32, [vp, i32, i32, vp, i64, vp, i32, i32, i32, i32, i32, vp, vp,
                                       i64, vp, i64, vp, vp, vp]),
        "fp8_requant_per_tensor": (i32, [vp, i64, vp, i32, i32, vp, vp, vp]),
        "fp8_requant_per_tensor_ex": (i32, [vp, i64, vp, i32, i32, i32, i32, vp, vp, vp, sz, vp]),
        "moe_status_sync": (i32, [vp, vp]),
        "moe_status_string": (C.c_char_p, [i32]),
        "moe_version": (C.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


def lib():
    return _lib if _lib is not None else load()


def _ptr(t):
    """Device address of a CUDA tensor (or a raw integer address, or None).
    A CPU tensor is rejected here: its host address would reach a kernel.
    Plain integers go to ctypes as they are (a void* argument accepts them)."""
    if t is None:
        return None
    if type(t) is int:
        return t
    if not t.is_cuda:
        raise ValueError(f"moeperm: tensor on {t.device}, but every tensor argument must be on "
                         "a CUDA device")
    return t.data_ptr()


# The current stream's raw handle without building a torch Stream object (the
# public call costs microseconds per launch on small problems); the public
# call is the fallback where these functions are absent.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream=None):
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None and _cur_device is not None:
        return _raw_stream(_cur_device())
    return torch.cuda.current_stream().cuda_stream


def _check(code: int, where: str):
    if code != MOE_OK:
        raise MoePermError(code, where)


# ---------------------------------------------------------------------------
# One-to-one C calls
# ---------------------------------------------------------------------------

def moe_compact_bound(A: int, L: int, block_e: int) -> int:
    return int(lib().moe_compact_bound(A, L, block_e))


def moe_should_use_masked(E: int, L: int) -> bool:
    return bool(lib().moe_should_use_masked(E, L))


def moe_scale_bytes(fmt: str, rows: int, H: int, g: int) -> int:
    return int(lib().moe_scale_bytes(FMT[fmt], rows, H, g))


def moe_workspace_bytes(T: int, K: int, L: int) -> int:
    return int(lib().moe_workspace_bytes(T, K, L))


def moe_dispatch_compact(x, ldx, T, d_num_tokens, H, topk_ids, topk_weights, K, E, L, block_e,
                         g, fmt, xq, scales, ld_s, m_indices, bound, src2dst, counts, starts,
                         psum, total, row_weights, workspace, workspace_bytes, d_status,
                         stream=None) -> int:
    return int(lib().moe_dispatch_compact(
        _ptr(x), ldx, T, _ptr(d_num_tokens), H, _ptr(topk_ids), _ptr(topk_weights), K, E, L,
        block_e, g, FMT[fmt], _ptr(xq), _ptr(scales), ld_s, _ptr(m_indices), bound,
        _ptr(src2dst), _ptr(counts), _ptr(starts), _ptr(psum), _ptr(total), _ptr(row_weights),
        _ptr(workspace), workspace_bytes, _ptr(d_status), _stream(stream)))


def moe_dispatch_compact_noalloc(x, ldx, T, d_num_tokens, H, topk_ids, topk_weights, K, E, L,
                                 block_e, g, fmt, xq, scales, ld_s, m_indices, bound, src2dst,
                                 counts, starts, psum, total, row_weights, d_status,
                                 stream=None) -> int:
    """moe_dispatch_compact for callers that cannot allocate device memory: the
    scratch is a static device array inside the library (see the C header)."""
    return int(lib().moe_dispatch_compact_noalloc(
        _ptr(x), ldx, T, _ptr(d_num_tokens), H, _ptr(topk_ids), _ptr(topk_weights), K, E, L,
        block_e, g, FMT[fmt], _ptr(xq), _ptr(scales), ld_s, _ptr(m_indices), bound,
        _ptr(src2dst), _ptr(counts), _ptr(starts), _ptr(psum), _ptr(total), _ptr(row_weights),
        _ptr(d_status), _stream(stream)))


def moe_dispatch_masked(x, ldx, T, d_num_tokens, H, topk_ids, topk_weights, K, E, L, cap, g,
                        fmt, xq, scales, ld_s, masked_m, src2dst, row_weights, psum, psum_align,
                        workspace, workspace_bytes, d_status, stream=None) -> int:
    return int(lib().moe_dispatch_masked(
        _ptr(x), ldx, T, _ptr(d_num_tokens), H, _ptr(topk_ids), _ptr(topk_weights), K, E, L,
        cap, g, FMT[fmt], _ptr(xq), _ptr(scales), ld_s, _ptr(masked_m), _ptr(src2dst),
        _ptr(row_weights), _ptr(psum), psum_align, _ptr(workspace), workspace_bytes,
        _ptr(d_status), _stream(stream)))


def moe_quant_group(x, ldx, T_cap, d_num_live, H, g, fmt, xq, scales, ld_s, d_status,
                    stream=None) -> int:
    return int(lib().moe_quant_group(_ptr(x), ldx, T_cap, _ptr(d_num_live), H, g, FMT[fmt],
                                      _ptr(xq), _ptr(scales), ld_s, _ptr(d_status),
                                      _stream(stream)))


def moe_combine(y, ldy, R, src2dst, w, T, d_num_tokens, K, H, out, d_status, stream=None) -> int:
    return int(lib().moe_combine(_ptr(y), ldy, R, _ptr(src2dst), _ptr(w), T, _ptr(d_num_tokens),
                                 K, H, _ptr(out), _ptr(d_status), _stream(stream)))


def moe_expand_to_slab(exp, elem_bytes, H, R, exp_scales, ld_es, psum, L, align, cap, fmt, g,
                       slab, slab_scales, ld_ss, masked_m, d_status, stream=None) -> int:
    return int(lib().moe_expand_to_slab(
        _ptr(exp), elem_bytes, H, R, _ptr(exp_scales), ld_es, _ptr(psum), L, align, cap,
        FMT[fmt], g, _ptr(slab), _ptr(slab_scales), ld_ss, _ptr(masked_m), _ptr(d_status),
        _stream(stream)))


def moe_expand_from_slab(slab, elem_bytes, H, slab_scales, ld_ss, psum, L, align, cap, fmt, g,
                         row_weights, exp, R, exp_scales, ld_es, m_indices, d_status,
                         stream=None) -> int:
    return int(lib().moe_expand_from_slab(
        _ptr(slab), elem_bytes, H, _ptr(slab_scales), ld_ss, _ptr(psum), L, align, cap,
        FMT[fmt], g, _ptr(row_weights), _ptr(exp), R, _ptr(exp_scales), ld_es, _ptr(m_indices),
        _ptr(d_status), _stream(stream)))


def fp8_requant_per_tensor(q, ldq, s_tok, T, H, q_out, d_scale_out, stream=None) -> int:
    return int(lib().fp8_requant_per_tensor(_ptr(q), ldq, _ptr(s_tok), T, H, _ptr(q_out),
                                            _ptr(d_scale_out), _stream(stream)))


TOKSCALE = {"f32": 0, "ue8m0": 1}
REQUANT_MODE = {"max_scale": 0, "amax": 1}


def fp8_requant_per_tensor_ex(q, ldq, s_tok, s_fmt, T, H, mode, q_out, d_scale_out, workspace,
                              workspace_bytes, stream=None) -> int:
    return int(lib().fp8_requant_per_tensor_ex(
        _ptr(q), ldq, _ptr(s_tok), TOKSCALE[s_fmt], T, H, REQUANT_MODE[mode], _ptr(q_out),
        _ptr(d_scale_out), _ptr(workspace), workspace_bytes, _stream(stream)))


def moe_status_sync(d_status, stream=None) -> int:
    return int(lib().moe_status_sync(_ptr(d_status), _stream(stream)))


def moe_version() -> str:
    return lib().moe_version().decode()


# ---------------------------------------------------------------------------
# Allocating helpers (torch owns the memory)
# ---------------------------------------------------------------------------

def scale_tensor(fmt: str, rows: int, H: int, g: int, device, blocks: int = 1, ld: int | None = None):
    """Allocate a scale tensor in `fmt`: u8 -> uint8 [rows, G]; f32pow2 -> float32
    [rows, G]; packed -> int32 [blocks, G4, ld] (ld = rows per block rounded up
    to 4). Returns (tensor, ld)."""
    G = H // g
    if fmt in ("u8", "mx"):
        ld = G if ld is None else ld
        return torch.empty((rows, ld), dtype=torch.uint8, device=device), ld
    if fmt in ("f32pow2", "f32"):
        ld = G if ld is None else ld
        return torch.empty((rows, ld), dtype=torch.float32, device=device), ld
    rpb = rows // blocks
    ld = (rpb + 3) // 4 * 4 if ld is None else ld
    return torch.empty((blocks, (G + 3) // 4, ld), dtype=torch.int32, device=device), ld


class Workspace:
    """Dispatch workspace, reusable across calls on one stream. Every dispatch
    writes the chunk table before reading it, so no initialisation is needed
    (no fill kernel per allocation)."""

    def __init__(self, T: int, K: int, L: int, device):
        self.nbytes = moe_workspace_bytes(T, K, L)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)

    def fits(self, T, K, L):
        return moe_workspace_bytes(T, K, L) <= self.nbytes


def dispatch_compact(x, topk_ids, topk_weights, num_experts, num_local_experts, block_e=128,
                     group_size=128, scale_fmt="packed", num_tokens=None, workspace=None,
                     status=None, row_weights=True):
    """Quantise + scatter into the compact layout. Returns a dict of tensors."""
    T, H = x.shape
    K = topk_ids.shape[1]
    L = num_local_experts
    dev = x.device
    bound = moe_compact_bound(T * K, L, block_e)
    xq = torch.empty((bound, H), dtype=torch.uint8, device=dev)
    sc, ld = scale_tensor(scale_fmt, bound, H, group_size, dev)
    out = dict(
        xq=xq, scales=sc, ld_s=ld, bound=bound,
        m_indices=torch.empty(bound, dtype=torch.int32, device=dev),
        src2dst=torch.empty((T, K), dtype=torch.int32, device=dev),
        counts=torch.empty(L, dtype=torch.int32, device=dev),
        starts=torch.empty(L, dtype=torch.int32, device=dev),
        psum=torch.empty(L, dtype=torch.int32, device=dev),
        total=torch.empty(1, dtype=torch.int32, device=dev),
        row_weights=torch.empty(bound, dtype=torch.float32, device=dev) if row_weights else None,
    )
    ws = workspace if workspace is not None else Workspace(T, K, L, dev)
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    code = moe_dispatch_compact(
        x, x.stride(0), T, num_tokens, H, topk_ids, topk_weights, K, num_experts, L, block_e,
        group_size, scale_fmt, xq, sc, ld, out["m_indices"], bound, out["src2dst"],
        out["counts"], out["starts"], out["psum"], out["total"], out["row_weights"], ws.buf,
        ws.nbytes, st)
    _check(code, "moe_dispatch_compact")
    out["status"] = st
    return out


def dispatch_masked(x, topk_ids, topk_weights, num_experts, num_local_experts, cap,
                    group_size=128, scale_fmt="packed", num_tokens=None, workspace=None,
                    status=None, row_weights=True, psum_align=128):
    """Quantise + scatter into per-expert slabs [L, cap, H]. Returns a dict,
    including psum [L], the expanded layout of the slab rows aligned to
    psum_align (None: not computed), and expand_rows, the static row count of
    that layout."""
    T, H = x.shape
    K = topk_ids.shape[1]
    L = num_local_experts
    dev = x.device
    xq = torch.empty((L, cap, H), dtype=torch.uint8, device=dev)
    sc, ld = scale_tensor(scale_fmt, L * cap, H, group_size, dev, blocks=L)
    out = dict(
        xq=xq, scales=sc, ld_s=ld,
        masked_m=torch.empty(L, dtype=torch.int32, device=dev),
        src2dst=torch.empty((T, K), dtype=torch.int32, device=dev),
        row_weights=torch.empty(L * cap, dtype=torch.float32, device=dev) if row_weights else None,
        psum=torch.empty(L, dtype=torch.int32, device=dev) if psum_align else None,
        expand_rows=moe_compact_bound(T * K, L, psum_align) if psum_align else 0,
    )
    ws = workspace if workspace is not None else Workspace(T, K, L, dev)
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    code = moe_dispatch_masked(
        x, x.stride(0), T, num_tokens, H, topk_ids, topk_weights, K, num_experts, L, cap,
        group_size, scale_fmt, xq, sc, ld, out["masked_m"], out["src2dst"], out["row_weights"],
        out["psum"], psum_align or 1, ws.buf, ws.nbytes, st)
    _check(code, "moe_dispatch_masked")
    out["status"] = st
    return out


def quant_group(x, group_size=128, scale_fmt="packed", num_live=None, status=None):
    """Quantise rows [0, num_live) of x (all rows when num_live is None)."""
    T_cap, H = x.shape
    dev = x.device
    xq = torch.empty((T_cap, H), dtype=torch.uint8, device=dev)
    sc, ld = scale_tensor(scale_fmt, T_cap, H, group_size, dev)
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    _check(moe_quant_group(x, x.stride(0), T_cap, num_live, H, group_size, scale_fmt, xq, sc, ld,
                           st), "moe_quant_group")
    return dict(xq=xq, scales=sc, ld_s=ld, status=st)


def combine(y, src2dst, weights=None, num_tokens=None, status=None, out=None):
    """out[t] = bf16(sum_k w[t,k] * y[src2dst[t,k]]) (fp32 accumulation)."""
    T, K = src2dst.shape
    R, H = y.shape
    dev = y.device
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if out is None else out
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    _check(moe_combine(y, y.stride(0), R, src2dst, weights, T, num_tokens, K, H, out, st),
           "moe_combine")
    return out


def expand_to_slab(exp, psum, num_local_experts, cap, align=128, exp_scales=None, ld_es=0,
                   scale_fmt="packed", group_size=128, status=None):
    """Expanded rows (e4m3 as uint8 / float8, or bfloat16 [R, H]) with segment
    ends psum [L] -> per-expert slabs [L, cap, H]; the scales follow when
    exp_scales is given. Returns a dict (slab, scales, ld_s, masked_m, status)."""
    R, H = exp.shape
    L = num_local_experts
    dev = exp.device
    slab = torch.empty((L, cap, H), dtype=exp.dtype, device=dev)
    ssc, ld_ss = (scale_tensor(scale_fmt, L * cap, H, group_size, dev, blocks=L)
                  if exp_scales is not None else (None, 0))
    masked_m = torch.empty(L, dtype=torch.int32, device=dev)
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    _check(moe_expand_to_slab(exp, exp.element_size(), H, R, exp_scales, ld_es, psum, L, align,
                              cap, scale_fmt, group_size, slab, ssc, ld_ss, masked_m, st),
           "moe_expand_to_slab")
    return dict(slab=slab, scales=ssc, ld_s=ld_ss, masked_m=masked_m, status=st)


def expand_from_slab(slab, psum, num_rows, align=128, slab_scales=None, ld_ss=0,
                     scale_fmt="packed", group_size=128, row_weights=None, status=None,
                     m_indices=True):
    """Per-expert slabs [L, cap, H] -> expanded rows [num_rows, H] at the
    segment ends psum [L]; bfloat16 rows are scaled by row_weights when given.
    Returns a dict (exp, scales, ld_s, m_indices, status)."""
    L, cap, H = slab.shape
    dev = slab.device
    exp = torch.empty((num_rows, H), dtype=slab.dtype, device=dev)
    esc, ld_es = (scale_tensor(scale_fmt, num_rows, H, group_size, dev)
                  if slab_scales is not None else (None, 0))
    mi = torch.empty(num_rows, dtype=torch.int32, device=dev) if m_indices else None
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    _check(moe_expand_from_slab(slab, slab.element_size(), H, slab_scales, ld_ss, psum, L, align,
                                cap, scale_fmt, group_size, row_weights, exp, num_rows, esc,
                                ld_es, mi, st), "moe_expand_from_slab")
    return dict(exp=exp, scales=esc, ld_s=ld_es, m_indices=mi, status=st)


def requant(q, s_tok, s_fmt="f32", mode="max_scale"):
    """Per-token -> per-tensor e4m3 requant. s_tok: fp32 [T] ("f32") or e8m0
    bytes [T] ("ue8m0"); mode "max_scale" (S = max s) or "amax" (S = max of
    s * row amax / 448). Returns (q_out uint8 [T,H], S [1] f32)."""
    T, H = q.shape
    q_out = torch.empty((T, H), dtype=torch.uint8, device=q.device)
    S = torch.empty(1, dtype=torch.float32, device=q.device)
    if s_fmt == "f32" and mode == "max_scale":
        _check(fp8_requant_per_tensor(q, q.stride(0), s_tok, T, H, q_out, S),
               "fp8_requant_per_tensor")
    else:
        ws = torch.empty(max(T, 1), dtype=torch.float32, device=q.device)
        _check(fp8_requant_per_tensor_ex(q, q.stride(0), s_tok, s_fmt, T, H, mode, q_out, S, ws,
                                         ws.numel() * 4), "fp8_requant_per_tensor_ex")
    return q_out, S
