"""fp64 CPU oracle for paged grouped-query attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline / reference
legs may import this package.  The product library never calls it, and it shares
no code with the CUDA path: the arithmetic lives in ``oracle.c`` (plain C,
double precision, the textbook definition written out loop by loop).

Functions take CPU tensors (torch or numpy) holding the same bf16 bit patterns the
GPU sees and return float64 results.  The 8-bit KV cache (E4M3 codes, one fp32 scale per
(token, KV head) row) has its own append and attention: ``kv_append_fp8``,
``attention_fp8``, with the codec ``e4m3_encode`` / ``e4m3_decode``.

The merged Q/K/V projection (page 1 §4.4.3) is ``qkv_project``; ``qkv_append`` adds the
append of its k and v (rounded once to bf16 by ``bf16_round``) to the cache, optionally after
the per-head RMS normalisation of q and k (``rms_norm_heads``; Qwen3's QK-norm, not on the
pages) and the rotary position embedding of q and k (``rope``; RoFormer's definition, not on
the pages) at each token's position (``token_positions``).

Parity status: every function here is pinned by the CPU tests in
``tests/test_oracle_pins.py``, ``tests/test_oracle_fp8.py``, ``tests/test_oracle_qkv.py``,
``tests/test_oracle_rope.py`` and ``tests/test_oracle_qknorm.py`` (closed forms, library
routines on tiny cases -- torch SDPA, torch's float8_e4m3fn -- invariants, the format's
error bound and a high-precision brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (-O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def load_library(path: str):
    """Load an oracle shared object (the default one, or a test-built variant)."""
    lib = ctypes.CDLL(path)
    i32p = ctypes.POINTER(ctypes.c_int32)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    ci = ctypes.c_int
    lib.oracle_kv_append.argtypes = [u16p, u16p, u16p, u16p, i32p, ci, ci, i32p, i32p, ci,
                                     ci, ci, ci]
    lib.oracle_kv_append.restype = ci
    lib.oracle_attention_rows.argtypes = [f64p, f64p, i32p, i32p, ci, u16p, u16p, u16p,
                                          i32p, ci, ci, i32p, i32p, ci, ci, ci, ci, ci,
                                          ctypes.c_double, ci]
    lib.oracle_attention_rows.restype = ci
    lib.oracle_paged_attention.argtypes = [f64p, f64p, u16p, u16p, u16p, i32p, ci, ci, i32p,
                                           i32p, ci, ci, ci, ci, ci, ctypes.c_double, ci]
    lib.oracle_paged_attention.restype = ci
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ci
    u8p = ctypes.POINTER(ctypes.c_uint8)
    f32p = ctypes.POINTER(ctypes.c_float)
    lib.oracle_e4m3_encode.argtypes = [f32p, u8p, ctypes.c_long]
    lib.oracle_e4m3_encode.restype = None
    lib.oracle_e4m3_decode.argtypes = [u8p, f64p, ctypes.c_long]
    lib.oracle_e4m3_decode.restype = None
    lib.oracle_kv_append_fp8.argtypes = [u8p, u8p, f32p, f32p, u16p, u16p, i32p, ci, ci, i32p, i32p,
                                         ci, ci, ci, ci]
    lib.oracle_kv_append_fp8.restype = ci
    lib.oracle_paged_attention_fp8.argtypes = [f64p, f64p, u16p, u8p, u8p, f32p, f32p, i32p, ci, ci,
                                               i32p, i32p, ci, ci, ci, ci, ci, ctypes.c_double, ci]
    lib.oracle_paged_attention_fp8.restype = ci
    lib.oracle_qkv_project.argtypes = [f64p, u16p, u16p, i32p, ci, ci, ci, ci, ci]
    lib.oracle_qkv_project.restype = ci
    lib.oracle_bf16_round.argtypes = [f64p, u16p, ctypes.c_long]
    lib.oracle_bf16_round.restype = None
    lib.oracle_token_positions.argtypes = [i32p, i32p, i32p, ci]
    lib.oracle_token_positions.restype = ci
    lib.oracle_rope.argtypes = [f64p, ci, ci, ci, ci, ci, i32p, ctypes.c_double]
    lib.oracle_rope.restype = ci
    lib.oracle_rms_norm_heads.argtypes = [f64p, ci, ci, ci, ci, ci, u16p, ctypes.c_double]
    lib.oracle_rms_norm_heads.restype = ci
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _bits(x) -> np.ndarray:
    """bf16 tensor (torch) or uint16 array -> contiguous uint16 numpy array of its bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch

    assert x.dtype == torch.bfloat16 and x.device.type == "cpu"
    return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(x) -> np.ndarray:
    if isinstance(x, (list, tuple)):
        x = np.asarray(x)
    if not isinstance(x, np.ndarray):
        x = x.cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _p(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def max_threads() -> int:
    return _load().oracle_max_threads()


def kv_append(k_pool, v_pool, k_new, v_new, block_table, cu_q_lens, seq_lens, *,
              block_size: int = 256, lib=None):
    """Return (k_pool', v_pool') as uint16 arrays: the pools after appending the new rows.

    k_pool/v_pool: [num_blocks, block_size, Hkv, D]; k_new/v_new: [total_tokens, Hkv, D].
    """
    kp = _bits(k_pool).copy()
    vp = _bits(v_pool).copy()
    kn, vn = _bits(k_new), _bits(v_new)
    bt, cu, sl = _i32(block_table), _i32(cu_q_lens), _i32(seq_lens)
    num_blocks, bs, hkv, d = kp.shape
    assert bs == block_size
    lib = lib or _load()
    rc = lib.oracle_kv_append(_p(kp, ctypes.c_uint16), _p(vp, ctypes.c_uint16),
                              _p(kn, ctypes.c_uint16), _p(vn, ctypes.c_uint16),
                              _p(bt, ctypes.c_int32), bt.shape[1], num_blocks,
                              _p(cu, ctypes.c_int32), _p(sl, ctypes.c_int32), len(sl),
                              hkv, d, bs)
    if rc:
        raise ValueError(f"oracle_kv_append rejected its input (code {rc})")
    return kp, vp


def attention(q, k_pool, v_pool, block_table, cu_q_lens, seq_lens, *, scale: float,
              rows=None, num_threads: int = 0, lib=None):
    """Paged causal GQA attention in fp64.

    q: [total_tokens, Hq, D] bf16; pools: [num_blocks, block_size, Hkv, D] bf16.
    rows: None for every (token, head), else a pair of int sequences (tokens, heads).
    Returns (out, lse) float64: out [T, Hq, D] and lse [T, Hq] for rows=None,
    else out [n, D] and lse [n].
    """
    qb, kb, vb = _bits(q), _bits(k_pool), _bits(v_pool)
    bt, cu, sl = _i32(block_table), _i32(cu_q_lens), _i32(seq_lens)
    t, hq, d = qb.shape
    num_blocks, bs, hkv, d2 = kb.shape
    assert d == d2 and vb.shape == kb.shape
    if bt.ndim == 1:
        bt = bt.reshape(len(sl), -1)
    lib = lib or _load()
    if rows is None:
        out = np.zeros((t, hq, d), np.float64)
        lse = np.zeros((t, hq), np.float64)
        rc = lib.oracle_paged_attention(_p(out, ctypes.c_double), _p(lse, ctypes.c_double),
                                        _p(qb, ctypes.c_uint16), _p(kb, ctypes.c_uint16),
                                        _p(vb, ctypes.c_uint16), _p(bt, ctypes.c_int32),
                                        bt.shape[1], num_blocks, _p(cu, ctypes.c_int32),
                                        _p(sl, ctypes.c_int32), len(sl), hq, hkv, d, bs,
                                        float(scale), int(num_threads))
    else:
        toks = _i32(np.asarray(rows[0]))
        hds = _i32(np.asarray(rows[1]))
        n = len(toks)
        out = np.zeros((n, d), np.float64)
        lse = np.zeros((n,), np.float64)
        rc = lib.oracle_attention_rows(_p(out, ctypes.c_double), _p(lse, ctypes.c_double),
                                       _p(toks, ctypes.c_int32), _p(hds, ctypes.c_int32), n,
                                       _p(qb, ctypes.c_uint16), _p(kb, ctypes.c_uint16),
                                       _p(vb, ctypes.c_uint16), _p(bt, ctypes.c_int32),
                                       bt.shape[1], num_blocks, _p(cu, ctypes.c_int32),
                                       _p(sl, ctypes.c_int32), len(sl), hq, hkv, d, bs,
                                       float(scale), int(num_threads))
    if rc:
        raise ValueError(f"oracle attention rejected its input (code {rc})")
    return out, lse


# ------------------------------------------------------------------ 8-bit KV cache

def _u8(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.cpu().numpy()
    assert x.dtype == np.uint8
    return np.ascontiguousarray(x)


def _f32(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def e4m3_encode(x, *, lib=None) -> np.ndarray:
    """float32 values -> E4M3 codes (round to nearest even, |x| > 448 -> +-448)."""
    xf = _f32(np.asarray(x, dtype=np.float32))
    out = np.zeros(xf.shape, np.uint8)
    (lib or _load()).oracle_e4m3_encode(_p(xf, ctypes.c_float), _p(out, ctypes.c_uint8), xf.size)
    return out


def e4m3_decode(c, *, lib=None) -> np.ndarray:
    """E4M3 codes -> float64 values."""
    cu = _u8(np.asarray(c, dtype=np.uint8))
    out = np.zeros(cu.shape, np.float64)
    (lib or _load()).oracle_e4m3_decode(_p(cu, ctypes.c_uint8), _p(out, ctypes.c_double), cu.size)
    return out


def kv_append_fp8(k_codes, v_codes, k_scale, v_scale, k_new, v_new, block_table, cu_q_lens,
                  seq_lens, *, block_size: int = 256, lib=None):
    """Return (k_codes', v_codes', k_scale', v_scale'): the 8-bit cache after quantising and
    appending the new rows.  codes: uint8 [num_blocks, block_size, Hkv, D]; scales: float32
    [num_blocks, Hkv, block_size]; k_new/v_new: bf16 [total_tokens, Hkv, D]."""
    kc, vc = _u8(k_codes).copy(), _u8(v_codes).copy()
    ks, vs = _f32(k_scale).copy(), _f32(v_scale).copy()
    kn, vn = _bits(k_new), _bits(v_new)
    bt, cu, sl = _i32(block_table), _i32(cu_q_lens), _i32(seq_lens)
    num_blocks, bs, hkv, d = kc.shape
    assert bs == block_size and ks.shape == (num_blocks, hkv, bs)
    rc = (lib or _load()).oracle_kv_append_fp8(
        _p(kc, ctypes.c_uint8), _p(vc, ctypes.c_uint8), _p(ks, ctypes.c_float), _p(vs, ctypes.c_float),
        _p(kn, ctypes.c_uint16), _p(vn, ctypes.c_uint16), _p(bt, ctypes.c_int32), bt.shape[1],
        num_blocks, _p(cu, ctypes.c_int32), _p(sl, ctypes.c_int32), len(sl), hkv, d, bs)
    if rc:
        raise ValueError(f"oracle_kv_append_fp8 rejected its input (code {rc})")
    return kc, vc, ks, vs


def attention_fp8(q, k_codes, v_codes, k_scale, v_scale, block_table, cu_q_lens, seq_lens, *,
                  scale: float, num_threads: int = 0, lib=None):
    """Paged causal GQA attention in fp64 over the 8-bit cache (K/V = code * row scale).
    Returns (out [T, Hq, D], lse [T, Hq]) float64."""
    qb = _bits(q)
    kc, vc, ks, vs = _u8(k_codes), _u8(v_codes), _f32(k_scale), _f32(v_scale)
    bt, cu, sl = _i32(block_table), _i32(cu_q_lens), _i32(seq_lens)
    t, hq, d = qb.shape
    num_blocks, bs, hkv, d2 = kc.shape
    assert d == d2 and vc.shape == kc.shape and ks.shape == (num_blocks, hkv, bs) == vs.shape
    if bt.ndim == 1:
        bt = bt.reshape(len(sl), -1)
    out = np.zeros((t, hq, d), np.float64)
    lse = np.zeros((t, hq), np.float64)
    if t:
        rc = (lib or _load()).oracle_paged_attention_fp8(
            _p(out, ctypes.c_double), _p(lse, ctypes.c_double), _p(qb, ctypes.c_uint16),
            _p(kc, ctypes.c_uint8), _p(vc, ctypes.c_uint8), _p(ks, ctypes.c_float), _p(vs, ctypes.c_float),
            _p(bt, ctypes.c_int32), bt.shape[1], num_blocks, _p(cu, ctypes.c_int32), _p(sl, ctypes.c_int32),
            len(sl), hq, hkv, d, bs, float(scale), int(num_threads))
        if rc:
            raise ValueError(f"oracle attention_fp8 rejected its input (code {rc})")
    return out, lse


Q_COLS, KV_COLS = 32 * 128, 8 * 128   # q: 32 heads, k and v: 8 KV heads, 128 dims each


def qkv_project(x, w, *, rows=None, num_threads: int = 0, lib=None) -> np.ndarray:
    """The merged projection y = x w^T in fp64 (page 1 §4.4.3 QKV fusion).

    x: [tokens, hidden] bf16; w: [n_out, hidden] bf16 (a linear layer's weight).  Returns
    y [len(rows) or tokens, n_out] float64 for the listed token rows (default: all).
    """
    xb, wb = _bits(x), _bits(w)
    tokens, hidden = xb.shape
    n_out, hw = wb.shape
    assert hw == hidden
    r = None if rows is None else _i32(np.asarray(rows))
    n_rows = tokens if r is None else len(r)
    y = np.zeros((n_rows, n_out), dtype=np.float64)
    lib = lib or _load()
    rc = lib.oracle_qkv_project(_p(y, ctypes.c_double), _p(xb, ctypes.c_uint16), _p(wb, ctypes.c_uint16),
                                None if r is None else _p(r, ctypes.c_int32), n_rows, tokens, hidden, n_out,
                                num_threads)
    if rc:
        raise ValueError(f"oracle_qkv_project rejected its input (code {rc})")
    return y


def bf16_round(v, *, lib=None) -> np.ndarray:
    """float64 values -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    out = np.zeros(a.shape, dtype=np.uint16)
    (lib or _load()).oracle_bf16_round(_p(a, ctypes.c_double), _p(out, ctypes.c_uint16), a.size)
    return out


def token_positions(cu_q_lens, seq_lens, *, lib=None) -> np.ndarray:
    """Absolute position of every new token (seq_len - q_len + i), int32 [total_tokens]."""
    cu, sl = _i32(cu_q_lens), _i32(seq_lens)
    pos = np.zeros(int(cu[-1]) if len(cu) else 0, dtype=np.int32)
    rc = (lib or _load()).oracle_token_positions(_p(pos, ctypes.c_int32), _p(cu, ctypes.c_int32),
                                                 _p(sl, ctypes.c_int32), len(sl))
    if rc:
        raise ValueError(f"oracle_token_positions rejected its input (code {rc})")
    return pos


def rope(y, positions, theta: float, *, first_col: int = 0, n_heads: int = 1, head_dim: int = 128,
         lib=None) -> np.ndarray:
    """Rotary position embedding (RoFormer, rotate-half pairing) of n_heads head vectors of
    each row of y from column first_col on, row t at positions[t]; returns a rotated copy."""
    out = np.array(y, dtype=np.float64, copy=True, order="C")
    if out.ndim == 1:
        out = out.reshape(1, -1)
    pos = _i32(np.asarray(positions))
    assert len(pos) == out.shape[0]
    rc = (lib or _load()).oracle_rope(_p(out, ctypes.c_double), out.shape[0], out.shape[1], first_col, n_heads,
                                      head_dim, _p(pos, ctypes.c_int32), float(theta))
    if rc:
        raise ValueError(f"oracle_rope rejected its input (code {rc})")
    return out


def rms_norm_heads(y, gain, eps: float, *, first_col: int = 0, n_heads: int = 1, head_dim: int = 128,
                   lib=None) -> np.ndarray:
    """Per-head RMS normalisation (QK-norm: RMSNorm of each head vector with the bf16 gain
    [head_dim], eps inside the square root) of n_heads head vectors of each row of y from
    column first_col on; returns a normalised copy."""
    out = np.array(y, dtype=np.float64, copy=True, order="C")
    if out.ndim == 1:
        out = out.reshape(1, -1)
    g = _bits(gain).reshape(-1)
    assert g.size == head_dim
    rc = (lib or _load()).oracle_rms_norm_heads(_p(out, ctypes.c_double), out.shape[0], out.shape[1], first_col,
                                                n_heads, head_dim, _p(g, ctypes.c_uint16), float(eps))
    if rc:
        raise ValueError(f"oracle_rms_norm_heads rejected its input (code {rc})")
    return out


def _bf16_values(v, lib=None) -> np.ndarray:
    """float64 values rounded to bf16 and widened back (exact)."""
    bits = bf16_round(v, lib=lib).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def qkv_append(x, w, k_pool, v_pool, block_table, cu_q_lens, seq_lens, *, rope_theta: float = 0.0,
               q_norm=None, k_norm=None, norm_eps: float = 1e-6, num_threads: int = 0, lib=None):
    """The merged projection of every new token with its k and v appended to the cache.

    Returns (q [tokens, 32, 128] float64, k_pool', v_pool' uint16): q is exact; the cache
    holds k and v rounded once to bf16 (its format), placed by ``kv_append``'s rule.  With
    q_norm and k_norm (bf16 gains [128]) the q and k columns are rounded to bf16 (the
    projection's output format) and every q head and k head is normalised (``rms_norm_heads``,
    eps norm_eps) before the rotation.  With rope_theta > 0 the 32 q heads and the 8 k heads of
    each token are then rotated at the token's absolute position (``rope``); v is never
    normalised or rotated.
    """
    y = qkv_project(x, w, num_threads=num_threads, lib=lib)
    t = y.shape[0]
    assert y.shape[1] == Q_COLS + 2 * KV_COLS
    assert (q_norm is None) == (k_norm is None), "QK-norm takes both gains"
    if q_norm is not None:
        y[:, :Q_COLS + KV_COLS] = _bf16_values(y[:, :Q_COLS + KV_COLS], lib=lib)
        y = rms_norm_heads(y, q_norm, norm_eps, first_col=0, n_heads=32, lib=lib)
        y = rms_norm_heads(y, k_norm, norm_eps, first_col=Q_COLS, n_heads=8, lib=lib)
    if rope_theta:
        pos = token_positions(cu_q_lens, seq_lens, lib=lib)
        y = rope(y, pos, rope_theta, first_col=0, n_heads=32, lib=lib)
        y = rope(y, pos, rope_theta, first_col=Q_COLS, n_heads=8, lib=lib)
    q = y[:, :Q_COLS].reshape(t, 32, 128)
    k_new = bf16_round(y[:, Q_COLS:Q_COLS + KV_COLS], lib=lib).reshape(t, 8, 128)
    v_new = bf16_round(y[:, Q_COLS + KV_COLS:], lib=lib).reshape(t, 8, 128)
    kp, vp = kv_append(k_pool, v_pool, k_new, v_new, block_table, cu_q_lens, seq_lens, lib=lib)
    return q, kp, vp
