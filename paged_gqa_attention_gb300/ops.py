"""Thin ctypes binding over libpagedattn.so (the C ABI in include/pagedattn.h).

Argument marshalling only: dtype/shape/device checks, raw pointers and the current
CUDA stream go to the library, which does every step of the computation in its own
sm_103a kernels.  PyTorch supplies device memory and streams.  There is no fallback:
if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedattn.so")

NUM_Q_HEADS, NUM_KV_HEADS, HEAD_DIM, BLOCK_SIZE = 32, 8, 128, 256
DEFAULT_SCALE = 1.0 / math.sqrt(HEAD_DIM)

STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_CUDA",
          4: "PA_ERR_DEVICE", 5: "PA_ERR_TIMEOUT", 6: "PA_ERR_WORKSPACE"}


class PagedAttnError(RuntimeError):
    """A library call returned a status other than PA_OK."""

    def __init__(self, fn: str, status: int, detail: int | None = None):
        self.status = status
        self.detail = detail
        msg = f"{fn}: {STATUS.get(status, status)}"
        if detail is not None:
            msg += f" (error word 0x{detail:x})"
        super().__init__(msg)


class pa_shape(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32)]


SHAPE = pa_shape(NUM_Q_HEADS, NUM_KV_HEADS, HEAD_DIM, BLOCK_SIZE)

_lib = None


def library_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load libpagedattn.so (built by paged_gqa_attention_gb300.build); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                           "`python -m paged_gqa_attention_gb300.build` (no fallback exists)")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, sz, i32, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_float
    u32p = ctypes.POINTER(ctypes.c_uint32)
    lib.pa_status_string.argtypes = [ctypes.c_int]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_version.argtypes = []
    lib.pa_version.restype = i32
    lib.pa_workspace_bytes.argtypes = [pa_shape, i32, i32]
    lib.pa_workspace_bytes.restype = sz
    lib.pa_workspace_init.argtypes = [vp, sz, vp]
    lib.pa_workspace_init.restype = ctypes.c_int
    lib.pa_check_error.argtypes = [vp, vp, u32p]
    lib.pa_check_error.restype = ctypes.c_int
    lib.kv_append.argtypes = [pa_shape, vp, vp, vp, vp, vp, i32, i32, vp, vp, i32, i32, vp, sz, vp]
    lib.kv_append.restype = ctypes.c_int
    lib.paged_qkv_append.argtypes = [pa_shape, i32, ctypes.c_float, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, i32, i32,
                                     vp, sz,
                                     vp]
    lib.paged_qkv_append.restype = ctypes.c_int
    lib.paged_qkv_append_qknorm.argtypes = [pa_shape, i32, ctypes.c_float, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp,
                                            vp, i32, i32, vp, vp, i32, i32, vp, sz, vp]
    lib.paged_qkv_append_qknorm.restype = ctypes.c_int
    lib.paged_attn_decode.argtypes = [pa_shape, vp, vp, vp, vp, vp, vp, i32, i32, vp, i32, f32, vp,
                                      sz, vp]
    lib.paged_attn_decode.restype = ctypes.c_int
    lib.paged_attn_decode_split.argtypes = [pa_shape, vp, vp, vp, vp, vp, vp, i32, i32, vp, i32,
                                            f32, i32, vp, sz, vp]
    lib.paged_attn_decode_split.restype = ctypes.c_int
    lib.paged_attn_decode_append.argtypes = [pa_shape, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp,
                                             i32, f32, vp, sz, vp]
    lib.paged_attn_decode_append.restype = ctypes.c_int
    lib.paged_attn_prefill.argtypes = [pa_shape, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, i32, i32,
                                       i32, f32, vp, sz, vp]
    lib.paged_attn_prefill.restype = ctypes.c_int
    lib.paged_attn_prefill_append.argtypes = [pa_shape, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, i32, i32,
                                              i32, f32, vp, sz, vp]
    lib.paged_attn_prefill_append.restype = ctypes.c_int
    lib.pa_decode_step_host_staging_bytes.argtypes = [pa_shape, i32, i32]
    lib.pa_decode_step_host_staging_bytes.restype = sz
    lib.pa_decode_step_host.argtypes = [pa_shape, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, i32, f32,
                                        vp, sz, vp, sz, vp]
    lib.pa_decode_step_host.restype = ctypes.c_int
    lib.kv_append_fp8.argtypes = [pa_shape, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, i32, i32, vp,
                                  sz, vp]
    lib.kv_append_fp8.restype = ctypes.c_int
    lib.paged_attn_decode_fp8.argtypes = [pa_shape, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, i32, f32,
                                          vp, sz, vp]
    lib.paged_attn_decode_fp8.restype = ctypes.c_int
    lib.paged_attn_decode_append_fp8.argtypes = [pa_shape, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                                 vp, i32, f32, vp, sz, vp]
    lib.paged_attn_decode_append_fp8.restype = ctypes.c_int
    lib.paged_attn_decode_fp8_split.argtypes = [pa_shape, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, i32,
                                                f32, i32, vp, sz, vp]
    lib.paged_attn_decode_fp8_split.restype = ctypes.c_int
    lib.pa_cascade_workspace_bytes.argtypes = [pa_shape, i32, i32, i32]
    lib.pa_cascade_workspace_bytes.restype = sz
    lib.paged_attn_decode_cascade.argtypes = [pa_shape, vp, vp, vp, vp, vp, vp, i32, i32, vp, i32, i32, f32,
                                              vp, sz, vp]
    lib.paged_attn_decode_cascade.restype = ctypes.c_int
    lib.pa_decode_graph_create.argtypes = [pa_shape, i32, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp,
                                           i32, f32, vp, sz, ctypes.POINTER(vp)]
    lib.pa_decode_graph_create.restype = ctypes.c_int
    lib.pa_decode_graph_launch.argtypes = [vp, vp]
    lib.pa_decode_graph_launch.restype = ctypes.c_int
    lib.pa_decode_graph_destroy.argtypes = [vp]
    lib.pa_decode_graph_destroy.restype = ctypes.c_int
    lib.pa_selftest_wait_timeout.argtypes = [vp, sz, ctypes.c_uint32, vp]
    lib.pa_selftest_wait_timeout.restype = ctypes.c_int
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != 0:
        raise PagedAttnError(fn, status)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None:
        for i, (a, b) in enumerate(zip(t.shape, shape)):
            if b is not None and a != b:
                raise ValueError(f"{name} has shape {tuple(t.shape)}, dim {i} must be {b}")
        if len(t.shape) != len(shape):
            raise ValueError(f"{name} must have {len(shape)} dims, got {tuple(t.shape)}")


# ------------------------------------------------------------------ workspace

def workspace_bytes(max_batch: int, max_blocks_per_seq: int) -> int:
    n = load().pa_workspace_bytes(SHAPE, int(max_batch), int(max_blocks_per_seq))
    if n == 0:
        raise ValueError("unsupported workspace request")
    return int(n)


def make_workspace(max_batch: int, max_blocks_per_seq: int, device=None, stream=None) -> torch.Tensor:
    """Allocate (with PyTorch) and zero (with pa_workspace_init) a workspace."""
    n = workspace_bytes(max_batch, max_blocks_per_seq)
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    _check("pa_workspace_init", load().pa_workspace_init(ws.data_ptr(), n, _stream(stream)))
    return ws


def check_error(workspace: torch.Tensor, stream=None) -> None:
    """Synchronise, read and clear the device error word; raise PagedAttnError if set."""
    word = ctypes.c_uint32(0)
    st = load().pa_check_error(workspace.data_ptr(), _stream(stream), ctypes.byref(word))
    if st != 0:
        raise PagedAttnError("pa_check_error", st, word.value)


# ------------------------------------------------------------------ the three calls

def kv_append(k_pool, v_pool, k_new, v_new, block_table, cu_q_lens, seq_lens, workspace,
              stream=None) -> None:
    """Write k_new/v_new [T, 8, 128] into the pools at each sequence's tail positions."""
    dev = k_pool.device
    _need(k_pool, "k_pool", torch.bfloat16, (None, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_pool, "v_pool", torch.bfloat16, tuple(k_pool.shape), dev)
    _need(k_new, "k_new", torch.bfloat16, (None, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_new, "v_new", torch.bfloat16, tuple(k_new.shape), dev)
    _need(block_table, "block_table", torch.int32, (None, None), dev)
    num_seqs = block_table.shape[0]
    _need(cu_q_lens, "cu_q_lens", torch.int32, (num_seqs + 1,), dev)
    _need(seq_lens, "seq_lens", torch.int32, (num_seqs,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    st = load().kv_append(SHAPE, k_pool.data_ptr(), v_pool.data_ptr(), k_new.data_ptr(),
                          v_new.data_ptr(), block_table.data_ptr(), block_table.shape[1],
                          k_pool.shape[0], cu_q_lens.data_ptr(), seq_lens.data_ptr(), num_seqs,
                          k_new.shape[0], workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check("kv_append", st)


QKV_COLS = NUM_Q_HEADS * HEAD_DIM + 2 * NUM_KV_HEADS * HEAD_DIM   # 6144


QWEN3_ROPE_THETA = 1.0e6
# Qwen3's eps inside the square root of its RMS normalisation (QK-norm)
QWEN3_NORM_EPS = 1.0e-6


def paged_qkv_append(x, w_qkv, k_pool, v_pool, block_table, cu_q_lens, seq_lens, workspace, *,
                     rope_theta: float = 0.0, q_norm_weight=None, k_norm_weight=None,
                     norm_eps: float = QWEN3_NORM_EPS, q_out=None, stream=None) -> torch.Tensor:
    """Merged Q/K/V projection of the new tokens: x [T, hidden] @ w_qkv[6144, hidden]^T; returns
    q [T, 32, 128] and writes k and v into the pools at each sequence's tail positions.
    rope_theta > 1 rotates the q and k heads at each token's position first (0: no rotation).
    q_norm_weight / k_norm_weight (bf16 [128], both or neither) normalise every q and k head by
    its RMS before the rotation (QK-norm, eps norm_eps; paged_qkv_append_qknorm)."""
    dev = x.device
    _need(x, "x", torch.bfloat16, (None, None), dev)
    hidden = x.shape[1]
    _need(w_qkv, "w_qkv", torch.bfloat16, (QKV_COLS, hidden), dev)
    _need(k_pool, "k_pool", torch.bfloat16, (None, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_pool, "v_pool", torch.bfloat16, tuple(k_pool.shape), dev)
    _need(block_table, "block_table", torch.int32, (None, None), dev)
    num_seqs = block_table.shape[0]
    _need(cu_q_lens, "cu_q_lens", torch.int32, (num_seqs + 1,), dev)
    _need(seq_lens, "seq_lens", torch.int32, (num_seqs,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    if q_out is None:
        q_out = torch.empty(x.shape[0], NUM_Q_HEADS, HEAD_DIM, dtype=torch.bfloat16, device=dev)
    _need(q_out, "q_out", torch.bfloat16, (x.shape[0], NUM_Q_HEADS, HEAD_DIM), dev)
    if (q_norm_weight is None) != (k_norm_weight is None):
        raise ValueError("QK-norm takes both q_norm_weight and k_norm_weight")
    if q_norm_weight is None:
        st = load().paged_qkv_append(SHAPE, hidden, float(rope_theta), q_out.data_ptr(), x.data_ptr(),
                                     w_qkv.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(), block_table.data_ptr(),
                                     block_table.shape[1], k_pool.shape[0], cu_q_lens.data_ptr(),
                                     seq_lens.data_ptr(), num_seqs, x.shape[0], workspace.data_ptr(),
                                     workspace.numel(), _stream(stream))
        _check("paged_qkv_append", st)
        return q_out
    _need(q_norm_weight, "q_norm_weight", torch.bfloat16, (HEAD_DIM,), dev)
    _need(k_norm_weight, "k_norm_weight", torch.bfloat16, (HEAD_DIM,), dev)
    st = load().paged_qkv_append_qknorm(SHAPE, hidden, float(rope_theta), q_norm_weight.data_ptr(),
                                        k_norm_weight.data_ptr(), float(norm_eps), q_out.data_ptr(), x.data_ptr(),
                                        w_qkv.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
                                        block_table.data_ptr(), block_table.shape[1], k_pool.shape[0],
                                        cu_q_lens.data_ptr(), seq_lens.data_ptr(), num_seqs, x.shape[0],
                                        workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check("paged_qkv_append_qknorm", st)
    return q_out


def paged_attn_decode(q, k_pool, v_pool, block_table, seq_lens, workspace, *,
                      scale: float = DEFAULT_SCALE, out=None, lse=None, split_tokens: int = 0,
                      stream=None) -> torch.Tensor:
    """One query token per sequence: q [B, 32, 128] -> out [B, 32, 128] (bf16).

    lse: optional fp32 [B, 32] tensor that receives the log-sum-exp of each row.
    split_tokens: context tokens per CTA (multiple of 64), 0 = the library's choice.
    """
    dev = q.device
    _need(q, "q", torch.bfloat16, (None, NUM_Q_HEADS, HEAD_DIM), dev)
    batch = q.shape[0]
    _need(k_pool, "k_pool", torch.bfloat16, (None, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_pool, "v_pool", torch.bfloat16, tuple(k_pool.shape), dev)
    _need(block_table, "block_table", torch.int32, (batch, None), dev)
    _need(seq_lens, "seq_lens", torch.int32, (batch,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, tuple(q.shape), dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, (batch, NUM_Q_HEADS), dev)
    lib = load()
    if split_tokens:
        st = lib.paged_attn_decode_split(SHAPE, out.data_ptr(), _ptr(lse), q.data_ptr(),
                                         k_pool.data_ptr(), v_pool.data_ptr(), block_table.data_ptr(),
                                         block_table.shape[1], k_pool.shape[0], seq_lens.data_ptr(),
                                         batch, float(scale), int(split_tokens), workspace.data_ptr(),
                                         workspace.numel(), _stream(stream))
    else:
        st = lib.paged_attn_decode(SHAPE, out.data_ptr(), _ptr(lse), q.data_ptr(), k_pool.data_ptr(),
                                   v_pool.data_ptr(), block_table.data_ptr(), block_table.shape[1],
                                   k_pool.shape[0], seq_lens.data_ptr(), batch, float(scale),
                                   workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check("paged_attn_decode", st)
    return out


def paged_attn_decode_append(q, k_new, v_new, k_pool, v_pool, block_table, seq_lens, workspace, *,
                             scale: float = DEFAULT_SCALE, out=None, lse=None,
                             stream=None) -> torch.Tensor:
    """kv_append of one new token per sequence (k_new/v_new [B, 8, 128], written at position
    seq_lens[b]-1) fused with paged_attn_decode: returns out [B, 32, 128]."""
    dev = q.device
    _need(q, "q", torch.bfloat16, (None, NUM_Q_HEADS, HEAD_DIM), dev)
    batch = q.shape[0]
    _need(k_new, "k_new", torch.bfloat16, (batch, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_new, "v_new", torch.bfloat16, (batch, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(k_pool, "k_pool", torch.bfloat16, (None, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_pool, "v_pool", torch.bfloat16, tuple(k_pool.shape), dev)
    _need(block_table, "block_table", torch.int32, (batch, None), dev)
    _need(seq_lens, "seq_lens", torch.int32, (batch,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, tuple(q.shape), dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, (batch, NUM_Q_HEADS), dev)
    st = load().paged_attn_decode_append(SHAPE, out.data_ptr(), _ptr(lse), q.data_ptr(),
                                         k_new.data_ptr(), v_new.data_ptr(), k_pool.data_ptr(),
                                         v_pool.data_ptr(), block_table.data_ptr(),
                                         block_table.shape[1], k_pool.shape[0], seq_lens.data_ptr(),
                                         batch, float(scale), workspace.data_ptr(), workspace.numel(),
                                         _stream(stream))
    _check("paged_attn_decode_append", st)
    return out


def fp8_cache(num_blocks: int, device=None):
    """An empty 8-bit KV cache: (k_codes, v_codes) uint8 [N, 256, 8, 128] holding the NaN code
    0x7F and (k_scale, v_scale) float32 [N, 8, 256] holding NaN, so a slot that was never
    written shows up as NaN wherever it is read."""
    dev = device or "cuda"
    codes = torch.full((num_blocks, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM), 0x7F, dtype=torch.uint8, device=dev)
    scales = torch.full((num_blocks, NUM_KV_HEADS, BLOCK_SIZE), float("nan"), dtype=torch.float32, device=dev)
    return codes, codes.clone(), scales, scales.clone()


def _need_fp8_cache(k_codes, v_codes, k_scale, v_scale, dev):
    _need(k_codes, "k_codes", torch.uint8, (None, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_codes, "v_codes", torch.uint8, tuple(k_codes.shape), dev)
    n = k_codes.shape[0]
    _need(k_scale, "k_scale", torch.float32, (n, NUM_KV_HEADS, BLOCK_SIZE), dev)
    _need(v_scale, "v_scale", torch.float32, (n, NUM_KV_HEADS, BLOCK_SIZE), dev)


def kv_append_fp8(k_codes, v_codes, k_scale, v_scale, k_new, v_new, block_table, cu_q_lens, seq_lens,
                  workspace, stream=None) -> None:
    """Quantise the new tokens' K/V rows into the 8-bit cache (in place)."""
    dev = k_new.device
    _need_fp8_cache(k_codes, v_codes, k_scale, v_scale, dev)
    _need(k_new, "k_new", torch.bfloat16, (None, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_new, "v_new", torch.bfloat16, tuple(k_new.shape), dev)
    _need(block_table, "block_table", torch.int32, (None, None), dev)
    num_seqs = block_table.shape[0]
    _need(cu_q_lens, "cu_q_lens", torch.int32, (num_seqs + 1,), dev)
    _need(seq_lens, "seq_lens", torch.int32, (num_seqs,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    st = load().kv_append_fp8(SHAPE, k_codes.data_ptr(), v_codes.data_ptr(), k_scale.data_ptr(),
                              v_scale.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), block_table.data_ptr(),
                              block_table.shape[1], k_codes.shape[0], cu_q_lens.data_ptr(),
                              seq_lens.data_ptr(), num_seqs, k_new.shape[0], workspace.data_ptr(),
                              workspace.numel(), _stream(stream))
    _check("kv_append_fp8", st)


def paged_attn_decode_fp8(q, k_codes, v_codes, k_scale, v_scale, block_table, seq_lens, workspace, *,
                          scale: float = DEFAULT_SCALE, out=None, lse=None, stream=None,
                          split_tokens: int = 0) -> torch.Tensor:
    """One query token per sequence over the 8-bit cache; returns out [B, 32, 128] bf16.
    split_tokens: context tokens per CTA (multiple of 64), 0 for the library's choice."""
    dev = q.device
    _need(q, "q", torch.bfloat16, (None, NUM_Q_HEADS, HEAD_DIM), dev)
    batch = q.shape[0]
    _need_fp8_cache(k_codes, v_codes, k_scale, v_scale, dev)
    _need(block_table, "block_table", torch.int32, (batch, None), dev)
    _need(seq_lens, "seq_lens", torch.int32, (batch,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, tuple(q.shape), dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, (batch, NUM_Q_HEADS), dev)
    st = load().paged_attn_decode_fp8_split(SHAPE, out.data_ptr(), _ptr(lse), q.data_ptr(), k_codes.data_ptr(),
                                            v_codes.data_ptr(), k_scale.data_ptr(), v_scale.data_ptr(),
                                            block_table.data_ptr(), block_table.shape[1], k_codes.shape[0],
                                            seq_lens.data_ptr(), batch, float(scale), int(split_tokens),
                                            workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check("paged_attn_decode_fp8", st)
    return out


def paged_attn_decode_append_fp8(q, k_new, v_new, k_codes, v_codes, k_scale, v_scale, block_table, seq_lens,
                                 workspace, *, scale: float = DEFAULT_SCALE, out=None, lse=None,
                                 stream=None) -> torch.Tensor:
    """kv_append_fp8 of one new token per sequence (k_new/v_new [B, 8, 128], written at
    position seq_lens[b]-1) fused with paged_attn_decode_fp8: returns out [B, 32, 128]."""
    dev = q.device
    _need(q, "q", torch.bfloat16, (None, NUM_Q_HEADS, HEAD_DIM), dev)
    batch = q.shape[0]
    _need(k_new, "k_new", torch.bfloat16, (batch, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_new, "v_new", torch.bfloat16, (batch, NUM_KV_HEADS, HEAD_DIM), dev)
    _need_fp8_cache(k_codes, v_codes, k_scale, v_scale, dev)
    _need(block_table, "block_table", torch.int32, (batch, None), dev)
    _need(seq_lens, "seq_lens", torch.int32, (batch,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, tuple(q.shape), dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, (batch, NUM_Q_HEADS), dev)
    st = load().paged_attn_decode_append_fp8(SHAPE, out.data_ptr(), _ptr(lse), q.data_ptr(), k_new.data_ptr(),
                                             v_new.data_ptr(), k_codes.data_ptr(), v_codes.data_ptr(),
                                             k_scale.data_ptr(), v_scale.data_ptr(), block_table.data_ptr(),
                                             block_table.shape[1], k_codes.shape[0], seq_lens.data_ptr(), batch,
                                             float(scale), workspace.data_ptr(), workspace.numel(),
                                             _stream(stream))
    _check("paged_attn_decode_append_fp8", st)
    return out


def make_cascade_workspace(max_batch: int, max_blocks_per_seq: int, shared_blocks: int, device=None,
                           stream=None) -> torch.Tensor:
    """Allocate and zero a workspace for paged_attn_decode_cascade."""
    n = load().pa_cascade_workspace_bytes(SHAPE, max_batch, max_blocks_per_seq, shared_blocks)
    if n == 0:
        raise ValueError("invalid cascade workspace request")
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    _check("pa_workspace_init", load().pa_workspace_init(ws.data_ptr(), n, _stream(stream)))
    return ws


def paged_attn_decode_cascade(q, k_pool, v_pool, block_table, seq_lens, shared_blocks: int, workspace, *,
                              scale: float = DEFAULT_SCALE, out=None, lse=None, stream=None) -> torch.Tensor:
    """paged_attn_decode for sequences whose first shared_blocks table entries are the same
    blocks: the shared prefix attended once for all queries, then each private suffix."""
    dev = q.device
    _need(q, "q", torch.bfloat16, (None, NUM_Q_HEADS, HEAD_DIM), dev)
    batch = q.shape[0]
    _need(k_pool, "k_pool", torch.bfloat16, (None, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_pool, "v_pool", torch.bfloat16, tuple(k_pool.shape), dev)
    _need(block_table, "block_table", torch.int32, (batch, None), dev)
    _need(seq_lens, "seq_lens", torch.int32, (batch,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, tuple(q.shape), dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, (batch, NUM_Q_HEADS), dev)
    st = load().paged_attn_decode_cascade(SHAPE, out.data_ptr(), _ptr(lse), q.data_ptr(), k_pool.data_ptr(),
                                          v_pool.data_ptr(), block_table.data_ptr(), block_table.shape[1],
                                          k_pool.shape[0], seq_lens.data_ptr(), batch, int(shared_blocks),
                                          float(scale), workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check("paged_attn_decode_cascade", st)
    return out


class DecodeGraph:
    """A decode step over several layers captured as one CUDA graph (pa_decode_graph_*).

    The graph holds the tensors' device pointers: update their contents in place between
    launches (new q / k_new / v_new, seq_lens + 1, grown block tables), never rebind them.
    The tensors are kept alive for as long as the handle is."""

    def __init__(self, handle: int, tensors: tuple):
        self._handle = handle
        self._tensors = tensors

    def launch(self, stream=None) -> None:
        if not self._handle:
            raise RuntimeError("DecodeGraph is closed")
        _check("pa_decode_graph_launch", load().pa_decode_graph_launch(self._handle, _stream(stream)))

    def close(self) -> None:
        if self._handle:
            h, self._handle = self._handle, None
            _check("pa_decode_graph_destroy", load().pa_decode_graph_destroy(h))
        self._tensors = ()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def decode_graph(q, k_new, v_new, k_pool, v_pool, block_table, seq_lens, workspace, *,
                 out, lse=None, scale: float = DEFAULT_SCALE) -> DecodeGraph:
    """Capture paged_attn_decode_append over L layers as one CUDA graph.  Layer-major
    tensors: q / out [L, B, 32, 128], k_new / v_new [L, B, 8, 128], pools
    [L, N, 256, 8, 128], lse [L, B, 32] or None; block_table [B, W] and seq_lens [B]
    are shared by every layer."""
    dev = q.device
    _need(q, "q", torch.bfloat16, (None, None, NUM_Q_HEADS, HEAD_DIM), dev)
    layers, batch = q.shape[0], q.shape[1]
    _need(k_new, "k_new", torch.bfloat16, (layers, batch, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_new, "v_new", torch.bfloat16, (layers, batch, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(k_pool, "k_pool", torch.bfloat16, (layers, None, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_pool, "v_pool", torch.bfloat16, tuple(k_pool.shape), dev)
    _need(out, "out", torch.bfloat16, tuple(q.shape), dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, (layers, batch, NUM_Q_HEADS), dev)
    _need(block_table, "block_table", torch.int32, (batch, None), dev)
    _need(seq_lens, "seq_lens", torch.int32, (batch,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    handle = ctypes.c_void_p(0)
    st = load().pa_decode_graph_create(SHAPE, layers, out.data_ptr(), _ptr(lse), q.data_ptr(),
                                       k_new.data_ptr(), v_new.data_ptr(), k_pool.data_ptr(),
                                       v_pool.data_ptr(), block_table.data_ptr(), block_table.shape[1],
                                       k_pool.shape[1], seq_lens.data_ptr(), batch, float(scale),
                                       workspace.data_ptr(), workspace.numel(), ctypes.byref(handle))
    _check("pa_decode_graph_create", st)
    return DecodeGraph(handle.value, (q, k_new, v_new, k_pool, v_pool, block_table, seq_lens, workspace,
                                      out, lse))


def paged_attn_prefill(q, k_pool, v_pool, block_table, cu_q_lens, seq_lens, max_q_len: int,
                       workspace, *, scale: float = DEFAULT_SCALE, out=None, lse=None,
                       stream=None) -> torch.Tensor:
    """Causal attention of each sequence's new tokens: q [T, 32, 128] -> out [T, 32, 128]."""
    dev = q.device
    _need(q, "q", torch.bfloat16, (None, NUM_Q_HEADS, HEAD_DIM), dev)
    _need(k_pool, "k_pool", torch.bfloat16, (None, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_pool, "v_pool", torch.bfloat16, tuple(k_pool.shape), dev)
    _need(block_table, "block_table", torch.int32, (None, None), dev)
    num_seqs = block_table.shape[0]
    _need(cu_q_lens, "cu_q_lens", torch.int32, (num_seqs + 1,), dev)
    _need(seq_lens, "seq_lens", torch.int32, (num_seqs,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, tuple(q.shape), dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, (q.shape[0], NUM_Q_HEADS), dev)
    st = load().paged_attn_prefill(SHAPE, out.data_ptr(), _ptr(lse), q.data_ptr(), k_pool.data_ptr(),
                                   v_pool.data_ptr(), block_table.data_ptr(), block_table.shape[1],
                                   k_pool.shape[0], cu_q_lens.data_ptr(), seq_lens.data_ptr(),
                                   num_seqs, q.shape[0], int(max_q_len), float(scale),
                                   workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check("paged_attn_prefill", st)
    return out


def paged_attn_prefill_append(q, k_new, v_new, k_pool, v_pool, block_table, cu_q_lens, seq_lens, max_q_len: int,
                              workspace, *, scale: float = DEFAULT_SCALE, out=None, lse=None,
                              stream=None) -> torch.Tensor:
    """kv_append of the new tokens' k_new / v_new [T, 8, 128] followed by the causal attention
    of q [T, 32, 128], in one kernel; returns out [T, 32, 128] and writes the pools."""
    dev = q.device
    _need(q, "q", torch.bfloat16, (None, NUM_Q_HEADS, HEAD_DIM), dev)
    _need(k_new, "k_new", torch.bfloat16, (q.shape[0], NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_new, "v_new", torch.bfloat16, (q.shape[0], NUM_KV_HEADS, HEAD_DIM), dev)
    _need(k_pool, "k_pool", torch.bfloat16, (None, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM), dev)
    _need(v_pool, "v_pool", torch.bfloat16, tuple(k_pool.shape), dev)
    _need(block_table, "block_table", torch.int32, (None, None), dev)
    num_seqs = block_table.shape[0]
    _need(cu_q_lens, "cu_q_lens", torch.int32, (num_seqs + 1,), dev)
    _need(seq_lens, "seq_lens", torch.int32, (num_seqs,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, tuple(q.shape), dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, (q.shape[0], NUM_Q_HEADS), dev)
    st = load().paged_attn_prefill_append(SHAPE, out.data_ptr(), _ptr(lse), q.data_ptr(), k_new.data_ptr(),
                                          v_new.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
                                          block_table.data_ptr(), block_table.shape[1], k_pool.shape[0],
                                          cu_q_lens.data_ptr(), seq_lens.data_ptr(), num_seqs, q.shape[0],
                                          int(max_q_len), float(scale), workspace.data_ptr(), workspace.numel(),
                                          _stream(stream))
    _check("paged_attn_prefill_append", st)
    return out


def decode_step_host_staging(max_batch: int, max_blocks_per_seq: int, device=None) -> torch.Tensor:
    """Device staging buffer for decode_step_host."""
    n = load().pa_decode_step_host_staging_bytes(SHAPE, int(max_batch), int(max_blocks_per_seq))
    if n == 0:
        raise ValueError("unsupported staging request")
    return torch.empty(int(n), dtype=torch.uint8, device=device or "cuda")


def decode_step_host(out_host, q_host, k_new_host, v_new_host, block_table_host, seq_lens_host,
                     k_pool, v_pool, staging, workspace, *, scale: float = DEFAULT_SCALE,
                     lse_host=None, stream=None) -> None:
    """One decode step from host tensors (pinned for asynchronous copies): copy the inputs
    in, append each sequence's new token and attend (one kernel), copy out [B, 32, 128]
    (and lse [B, 32]) back.  Asynchronous on the stream; synchronise before reading out_host."""
    batch = q_host.shape[0]
    for t, name in ((out_host, "out"), (q_host, "q"), (k_new_host, "k_new"), (v_new_host, "v_new"),
                    (block_table_host, "block_table"), (seq_lens_host, "seq_lens")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    if q_host.dtype != torch.bfloat16 or tuple(q_host.shape[1:]) != (NUM_Q_HEADS, HEAD_DIM):
        raise ValueError("q must be bf16 [B, 32, 128]")
    for t, name in ((k_new_host, "k_new"), (v_new_host, "v_new")):
        if t.dtype != torch.bfloat16 or tuple(t.shape) != (batch, NUM_KV_HEADS, HEAD_DIM):
            raise ValueError(f"{name} must be bf16 [B, 8, 128]")
    if out_host.dtype != torch.bfloat16 or tuple(out_host.shape) != tuple(q_host.shape):
        raise ValueError("out must be bf16 like q")
    if block_table_host.dtype != torch.int32 or block_table_host.shape[0] != batch:
        raise ValueError("block_table must be int32 [B, W]")
    if seq_lens_host.dtype != torch.int32 or tuple(seq_lens_host.shape) != (batch,):
        raise ValueError("seq_lens must be int32 [B]")
    if lse_host is not None and (lse_host.is_cuda or lse_host.dtype != torch.float32):
        raise ValueError("lse must be a host fp32 tensor [B, 32]")
    _need(k_pool, "k_pool", torch.bfloat16, (None, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM))
    _need(v_pool, "v_pool", torch.bfloat16, tuple(k_pool.shape), k_pool.device)
    _need(staging, "staging", torch.uint8, None, k_pool.device)
    _need(workspace, "workspace", torch.uint8, None, k_pool.device)
    st = load().pa_decode_step_host(SHAPE, out_host.data_ptr(), _ptr(lse_host), q_host.data_ptr(),
                                    k_new_host.data_ptr(), v_new_host.data_ptr(),
                                    block_table_host.data_ptr(), seq_lens_host.data_ptr(), batch,
                                    block_table_host.shape[1], k_pool.data_ptr(), v_pool.data_ptr(),
                                    k_pool.shape[0], float(scale), staging.data_ptr(), staging.numel(),
                                    workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check("pa_decode_step_host", st)


def selftest_wait_timeout(workspace: torch.Tensor, timeout_us: int = 20000, stream=None) -> None:
    """Launch the bounded-wait self-test kernel (it always times out by design)."""
    _check("pa_selftest_wait_timeout",
           load().pa_selftest_wait_timeout(workspace.data_ptr(), workspace.numel(),
                                           int(timeout_us), _stream(stream)))
