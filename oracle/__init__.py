"""CPU oracle for the MoE permute / FP8-quantise / combine / requantise path.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` may import this package. The product path
(``combine_fp8_quant_gb300``) never imports it and has no CPU fallback.

The arithmetic lives in ``moeperm_oracle.c`` (plain C, scalar loops, exact
double arithmetic where the definition is exact). This module only builds it
with gcc, loads it and marshals numpy arrays. It shares no code, header or
constant with the CUDA library.

Parity pins: every function here is pinned in ``tests/test_oracle_pins.py``
against the OCP E4M3 specification, closed forms, brute force on tiny inputs,
library routines, and the constants the SGLang pull-request digests print.

Parity unpinned (fixed by decision because the sources leave them open, so no
source can confirm them): the row order inside an expert segment (ascending
t*K + k), the exponent of an all-zero group (from max(amax, 1e-10)), the byte
order and pad bytes of the packed UE8M0 words (group 4w in the low byte, pads
zero), and the per-tensor scale of the requant (S = max of the per-token
scales). Everything downstream of these choices is pinned.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moeperm_oracle.c")
_HDR = os.path.join(_HERE, "moeperm_oracle.h")
_LIB = os.path.join(_HERE, "libmoeperm_oracle.so")

FMT = {"u8": 0, "packed": 1, "f32pow2": 2, "f32": 3, "mx": 4}
FMT["f32_pow2"] = 2
ST_OVERFLOW, ST_LIVE_OVERFLOW, ST_BAD_LAYOUT = 1, 2, 4

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no -ffast-math, no FP contraction)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            _declare(_lib)
    return _lib


def _p(a):
    """Pointer to a numpy array's data (None for None)."""
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return C.c_void_p(a.ctypes.data)


def _declare(L):
    vp, i32, i64, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_float
    sig = {
        "ref_e4m3_encode": (C.c_uint8, [C.c_double]),
        "ref_e4m3_decode": (C.c_double, [C.c_uint8]),
        "ref_e4m3_encode_array": (None, [vp, i64, vp]),
        "ref_e4m3_decode_array": (None, [vp, i64, vp]),
        "ref_group_exponent": (i32, [f32]),
        "ref_group_exponent_array": (None, [vp, i64, vp]),
        "ref_bf16_rne": (C.c_uint16, [f32]),
        "ref_compact_bound": (i64, [i64, i64, i64]),
        "ref_should_use_masked": (i32, [i64, i64]),
        "ref_quant_row": (None, [vp, i32, i32, vp, vp]),
        "ref_quant_row_fmt": (None, [vp, i32, i32, i32, vp, vp, vp]),
        "ref_mx_exponent_array": (None, [vp, i64, vp]),
        "ref_scale_bytes": (i64, [i32, i64, i32, i32]),
        "ref_quant_group": (i32, [vp, i64, i32, i32, i32, i32, i32, vp, vp, i64]),
        "ref_dispatch_compact": (i32, [vp, i64, i32, i32, i32, vp, vp, i32, i32, i32, i32, i32,
                                       vp, vp, i64, vp, i64, vp, vp, vp, vp, vp, vp]),
        "ref_dispatch_masked": (i32, [vp, i64, i32, i32, i32, vp, vp, i32, i32, i32, i32, i32,
                                      vp, vp, i64, vp, vp, vp, vp, i32]),
        "ref_combine_f64": (None, [vp, i64, vp, vp, i32, i32, i32, vp, vp]),
        "ref_combine_f32": (None, [vp, i64, vp, vp, i32, i32, i32, vp]),
        "ref_requant": (None, [vp, i64, vp, i32, i32, vp, vp]),
        "ref_requant_ex": (None, [vp, i64, vp, i32, i32, i32, i32, vp, vp]),
        "ref_expand_to_slab": (i32, [vp, i32, i32, i64, vp, i64, vp, i32, i32, i32, i32, i32,
                                     vp, vp, i64, vp]),
        "ref_expand_from_slab": (i32, [vp, i32, i32, vp, i64, vp, i32, i32, i32, i32, i32, vp,
                                       vp, i64, vp, i64, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


# ---------------------------------------------------------------------------
# Scalar / elementwise helpers
# ---------------------------------------------------------------------------

def e4m3_encode(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().ref_e4m3_encode_array(_p(v), v.size, _p(out))
    return out


def e4m3_decode(c) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().ref_e4m3_decode_array(_p(c), c.size, _p(out))
    return out


def group_exponent(amax) -> np.ndarray:
    a = np.ascontiguousarray(amax, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.int32)
    lib().ref_group_exponent_array(_p(a), a.size, _p(out))
    return out


def mx_exponent(amax) -> np.ndarray:
    a = np.ascontiguousarray(amax, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.int32)
    lib().ref_mx_exponent_array(_p(a), a.size, _p(out))
    return out


def quant_row_fmt(x_bits: np.ndarray, g: int, fmt: str):
    """(q bytes [H], scale bytes [G], scale values [G] float32) for any format."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    H = x.size
    q = np.empty(H, np.uint8)
    eb = np.empty(H // g, np.uint8)
    sv = np.empty(H // g, np.float32)
    lib().ref_quant_row_fmt(_p(x), H, g, FMT[fmt], _p(q), _p(eb), _p(sv))
    return q, eb, sv


def bf16_rne(f: float) -> int:
    return int(lib().ref_bf16_rne(float(f)))


def compact_bound(A: int, L: int, block_e: int) -> int:
    return int(lib().ref_compact_bound(A, L, block_e))


def should_use_masked(E: int, L: int) -> bool:
    return bool(lib().ref_should_use_masked(E, L))


def scale_bytes(fmt: str, rows: int, H: int, g: int) -> int:
    return int(lib().ref_scale_bytes(FMT[fmt], rows, H, g))


def quant_row(x_bits: np.ndarray, g: int):
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    H = x.size
    q = np.empty(H, np.uint8)
    eb = np.empty(H // g, np.uint8)
    lib().ref_quant_row(_p(x), H, g, _p(q), _p(eb))
    return q, eb


# ---------------------------------------------------------------------------
# Scale-buffer shapes (the oracle's own reading of the layouts)
# ---------------------------------------------------------------------------

def scale_buffer(fmt: str, rows: int, G: int, fill: int = 0xA5, ld: int | None = None,
                 blocks: int = 1):
    """Allocate a scale buffer of the given layout, filled with a sentinel.

    u8:     uint8 [rows, ld]       (ld >= G)
    f32:    float32 [rows, ld]     (ld >= G)
    packed: uint8 bytes of int32 words; `blocks` blocks of [G4, ld] words,
            ld >= rows-per-block, rounded up to 4 by default.
    Returns (array, ld).
    """
    if fmt in ("u8", "mx"):
        ld = G if ld is None else ld
        return np.full((rows, ld), fill, np.uint8), ld
    if fmt in ("f32", "f32pow2", "f32_pow2"):
        ld = G if ld is None else ld
        a = np.full((rows, ld), fill, np.uint32).view(np.float32)
        return a, ld
    rpb = rows // blocks
    ld = (rpb + 3) // 4 * 4 if ld is None else ld
    G4 = (G + 3) // 4
    return np.full((blocks * G4 * ld * 4,), fill, np.uint8), ld


# ---------------------------------------------------------------------------
# Path functions
# ---------------------------------------------------------------------------

def quant_group(x, T_cap, n_live, H, g, fmt, xq, scales, ld_s, ldx=None):
    ldx = H if ldx is None else ldx
    return int(lib().ref_quant_group(_p(x), ldx, T_cap, n_live, H, g, FMT[fmt], _p(xq),
                                     _p(scales), ld_s))


def dispatch_compact(x, T, n_live, H, ids, w, K, L, block_e, g, fmt, xq, scales, ld_s,
                     m_indices, bound, src2dst, counts, starts, psum, total,
                     row_weights=None, ldx=None):
    ldx = H if ldx is None else ldx
    return int(lib().ref_dispatch_compact(
        _p(x), ldx, T, n_live, H, _p(ids), _p(w), K, L, block_e, g, FMT[fmt], _p(xq),
        _p(scales), ld_s, _p(m_indices), bound, _p(src2dst), _p(counts), _p(starts),
        _p(psum), _p(total), _p(row_weights)))


def dispatch_masked(x, T, n_live, H, ids, w, K, L, cap, g, fmt, xq, scales, ld_s,
                    masked_m, src2dst, row_weights=None, ldx=None, psum=None, psum_align=128):
    ldx = H if ldx is None else ldx
    return int(lib().ref_dispatch_masked(
        _p(x), ldx, T, n_live, H, _p(ids), _p(w), K, L, cap, g, FMT[fmt], _p(xq),
        _p(scales), ld_s, _p(masked_m), _p(src2dst), _p(row_weights), _p(psum), psum_align))


def combine_f64(y, src2dst, w, T, K, H, ldy=None):
    ldy = H if ldy is None else ldy
    out = np.empty((T, H), np.float64)
    mass = np.empty((T, H), np.float64)
    lib().ref_combine_f64(_p(y), ldy, _p(src2dst), _p(w), T, K, H, _p(out), _p(mass))
    return out, mass


def combine_f32(y, src2dst, w, T, K, H, ldy=None):
    ldy = H if ldy is None else ldy
    out = np.empty((T, H), np.uint16)
    lib().ref_combine_f32(_p(y), ldy, _p(src2dst), _p(w), T, K, H, _p(out))
    return out


def requant(q, s_tok, T, H, ldq=None):
    ldq = H if ldq is None else ldq
    out = np.empty((T, H), np.uint8)
    S = np.zeros(1, np.float32)
    lib().ref_requant(_p(q), ldq, _p(s_tok), T, H, _p(out), _p(S))
    return out, float(S[0])


def requant_ex(q, s_tok, T, H, s_fmt="f32", mode="max_scale", ldq=None):
    """s_fmt: "f32" or "ue8m0" (uint8 bytes); mode: "max_scale" or "amax"."""
    ldq = H if ldq is None else ldq
    out = np.empty((T, H), np.uint8)
    S = np.zeros(1, np.float32)
    lib().ref_requant_ex(_p(q), ldq, _p(s_tok), {"f32": 0, "ue8m0": 1}[s_fmt], T, H,
                         {"max_scale": 0, "amax": 1}[mode], _p(out), _p(S))
    return out, float(S[0])


def expand_to_slab(exp, elem_bytes, H, R, exp_scales, ld_es, psum, L, align, cap, fmt, g,
                   slab, slab_scales, ld_ss, masked_m):
    return int(lib().ref_expand_to_slab(
        _p(exp), elem_bytes, H, R, _p(exp_scales), ld_es, _p(psum), L, align, cap,
        FMT[fmt], g, _p(slab), _p(slab_scales), ld_ss, _p(masked_m)))


def expand_from_slab(slab, elem_bytes, H, slab_scales, ld_ss, psum, L, align, cap, fmt, g,
                     row_weights, exp, R, exp_scales, ld_es, m_indices):
    return int(lib().ref_expand_from_slab(
        _p(slab), elem_bytes, H, _p(slab_scales), ld_ss, _p(psum), L, align, cap, FMT[fmt],
        g, _p(row_weights), _p(exp), R, _p(exp_scales), ld_es, _p(m_indices)))
