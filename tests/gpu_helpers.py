"""Helpers shared by the GPU parity tests (test side only)."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_attention_gb300 import build as pa_build
from paged_gqa_attention_gb300 import ops
from paged_gqa_attention_gb300 import workloads as wl

# Parity bar for bf16 outputs with fp32 accumulation: over a whole output tensor,
# max |gpu - ref| <= 1e-2 and ||gpu - ref||_2 / ||ref||_2 <= 5e-3.
MAX_ABS = 1e-2
REL_RMS = 5e-3
# lse = m + log(sum_j p~_j), where p~_j = bf16(p_j) are the same rounded weights the PV
# product uses (so the normalised weights sum to one).  bf16 keeps 8 significant bits (7
# stored, 1 implicit): between 1 and 2 its values are 2^-7 apart, so round-to-nearest
# changes a weight by up to half of that, a relative |d| <= 2^-8 (1 + 2^-8 rounds to 1).
# Hence the sum moves by at most 2^-8 relative and the log by at most
# log(1 + 2^-8) = 3.90e-3, reached when one weight dominates the sum; fp32 accumulation of
# the 128-term scores adds about 1e-4.  Bar: 4e-3 absolute.
LSE_ABS = 4e-3


def lib_ready():
    pa_build.build()
    return ops.load()


def to_cpu(t):
    return t.detach().to("cpu")


def errors(gpu_out: torch.Tensor, ref: np.ndarray):
    g = gpu_out.detach().float().cpu().double().numpy()
    diff = g - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300)) if diff.size else 0.0
    return max_abs, rel


# Realised errors of every comparison made in this process, in order: (what, kind, values).
# The session hook in conftest.py writes them out when PA_PARITY_REPORT names a file.
REPORT = []


def assert_close(gpu_out, ref, what=""):
    assert np.isfinite(gpu_out.detach().float().cpu().numpy()).all(), f"{what}: non-finite output"
    max_abs, rel = errors(gpu_out, ref)
    REPORT.append({"what": what, "kind": "out", "max_abs": max_abs, "rel_rms": rel,
                   "elements": int(np.asarray(ref).size)})
    assert max_abs <= MAX_ABS and rel <= REL_RMS, f"{what}: max_abs={max_abs:.3e} rel_rms={rel:.3e}"
    return max_abs, rel


def assert_lse_close(gpu_lse, ref, what=""):
    g = gpu_lse.detach().double().cpu().numpy()
    err = float(np.max(np.abs(g - ref))) if g.size else 0.0
    REPORT.append({"what": what, "kind": "lse", "max_abs": err, "elements": int(np.asarray(ref).size)})
    assert err <= LSE_ABS, f"{what}: lse max_abs={err:.3e}"


def oracle_attention(batch: wl.Batch, k_pool=None, v_pool=None, rows=None):
    """Oracle over a batch; pools default to the batch's own (copied to the host)."""
    kp = to_cpu(batch.k_pool) if k_pool is None else k_pool
    vp = to_cpu(batch.v_pool) if v_pool is None else v_pool
    return oracle.attention(to_cpu(batch.q), kp, vp, to_cpu(batch.block_table),
                            to_cpu(batch.cu_q_lens), to_cpu(batch.seq_lens), scale=wl.SCALE,
                            rows=rows)


def oracle_appended_pools(batch: wl.Batch):
    """The pools after the oracle's own append of the batch's new tokens (host arrays)."""
    kp, vp = oracle.kv_append(to_cpu(batch.k_pool), to_cpu(batch.v_pool), to_cpu(batch.k_new),
                              to_cpu(batch.v_new), to_cpu(batch.block_table), to_cpu(batch.cu_q_lens),
                              to_cpu(batch.seq_lens))
    return kp, vp


def workspace_for(batch: wl.Batch):
    return ops.make_workspace(max(batch.num_seqs, 1), batch.max_blocks_per_seq, device=batch.q.device)


gpu = pytest.mark.gpu
