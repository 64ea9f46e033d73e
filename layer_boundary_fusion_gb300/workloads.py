"""Seeded synthetic inputs for the layer-boundary workloads.

This module only draws numbers: it holds none of the boundary's arithmetic, and both
the CUDA path and the CPU oracle consume exactly the bf16 bit patterns it returns.
Arrays are numpy: bf16 tensors are ``uint16`` arrays of raw bf16 bits (rounded from
the drawn float32 values to nearest-even by torch's CPU cast), gamma and routing
weights are float32, indices int32.

Recipe (one independent PCG64 stream per tensor, keyed by (seed, stream id)):
  * partial contributions and residual rows: normal with the stated standard
    deviation;
  * gamma = 1 + 0.1 * N(0, 1), float32;
  * prefill outliers: round(1% of T) distinct rows, chosen by seeded sampling, are
    multiplied by 50 in every partial before the bf16 rounding;
  * ragged token sets: each set's rows are padded up to a multiple of 8 and the sets
    are concatenated; padding rows of every partial are zero;
  * MoE: logits N(0, 1) over the experts, top-k by value (ties to the lower expert
    id), routing weights = softmax over the chosen k (float64, stored as float32);
    the (token, slot) pairs are sorted stably by (expert, token, slot), and row p of
    the expert output belongs to the pair in sorted position p, so idx[t, j] = p.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

# stream ids: one independent generator per tensor
_S_PARTIAL = 0          # + k
_S_RESIDUAL = 100
_S_GAMMA = 200
_S_OUTLIER = 300
_S_LOGITS = 400
_S_EXPERT = 500


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> raw bf16 bits (round to nearest even, by torch's CPU cast)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def normal_bf16(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    x = _rng(seed, stream).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x = x * np.float32(std)
    return to_bf16_bits(x)


def gamma_f32(seed: int, H: int) -> np.ndarray:
    g = _rng(seed, _S_GAMMA).standard_normal(H, dtype=np.float32)
    return (np.float32(1.0) + np.float32(0.1) * g).astype(np.float32)


@dataclasses.dataclass
class Workload:
    name: str
    T: int                      # rows the call processes (S for a slice)
    H: int
    eps: float
    gamma: np.ndarray
    residual: Optional[np.ndarray]          # bf16 bits [T,H] (or [S,H] for a slice)
    partials: List[np.ndarray] = dataclasses.field(default_factory=list)
    fp8: bool = False
    # ragged row slice
    T_pad: int = 0
    num_slices: int = 1
    slice: int = 0
    set_offsets: Optional[np.ndarray] = None     # int32 [num_sets]
    set_counts: Optional[np.ndarray] = None      # int32 [num_sets]
    residual_full: Optional[np.ndarray] = None   # bf16 [T_pad,H], slice rows = residual
    # MoE finalize
    expert_out: Optional[np.ndarray] = None      # bf16 bits [T*topk, H], expert-sorted
    idx: Optional[np.ndarray] = None             # int32 [T, topk]
    w: Optional[np.ndarray] = None               # float32 [T, topk]
    topk: int = 0
    num_experts: int = 0

    @property
    def K(self) -> int:
        return len(self.partials)


def fold_workload(name, K, T, H, seed, *, partial_std=1.0, residual=True,
                  residual_std=1.0, eps=1e-6, outlier_frac=0.0, outlier_scale=50.0,
                  fp8=False) -> Workload:
    """K partial buffers [T,H] plus a residual [T,H] (None for the Initial state)."""
    outlier_rows = np.zeros(0, np.int64)
    if outlier_frac > 0.0:
        n_out = int(round(outlier_frac * T))
        outlier_rows = np.sort(_rng(seed, _S_OUTLIER).choice(T, size=n_out, replace=False))
    partials = []
    for k in range(K):
        x = _rng(seed, _S_PARTIAL + k).standard_normal((T, H), dtype=np.float32)
        if partial_std != 1.0:
            x = x * np.float32(partial_std)
        if outlier_rows.size:
            x[outlier_rows] *= np.float32(outlier_scale)
        partials.append(to_bf16_bits(x))
    res = normal_bf16(seed, _S_RESIDUAL, (T, H), residual_std) if residual else None
    return Workload(name=name, T=T, H=H, eps=eps, gamma=gamma_f32(seed, H),
                    residual=res, partials=partials, fp8=fp8)


def ragged_layout(counts, pad_multiple=8):
    """Padded offsets of token sets concatenated in the given order, and T_pad."""
    offsets, off = [], 0
    for c in counts:
        offsets.append(off)
        off += -(-int(c) // pad_multiple) * pad_multiple
    return np.asarray(offsets, np.int32), np.asarray(counts, np.int32), off


def slice_workload(name, K, H, counts, num_slices, slice_, seed, *, eps=1e-6,
                   fp8=False) -> Workload:
    """K partial buffers over a padded ragged batch (padding rows zero) and the
    compact [S,H] residual of one slice; residual_full holds every slice's rows."""
    offsets, counts, T_pad = ragged_layout(counts)
    valid = np.zeros(T_pad, bool)
    for o, c in zip(offsets, counts):
        valid[o:o + c] = True
    partials = []
    for k in range(K):
        x = _rng(seed, _S_PARTIAL + k).standard_normal((T_pad, H), dtype=np.float32)
        x[~valid] = 0.0
        partials.append(to_bf16_bits(x))
    full = _rng(seed, _S_RESIDUAL).standard_normal((T_pad, H), dtype=np.float32)
    full[~valid] = 0.0
    residual_full = to_bf16_bits(full)
    S = T_pad // num_slices
    return Workload(name=name, T=S, H=H, eps=eps, gamma=gamma_f32(seed, H),
                    residual=residual_full[slice_ * S:(slice_ + 1) * S].copy(),
                    partials=partials, fp8=fp8, T_pad=T_pad, num_slices=num_slices,
                    slice=slice_, set_offsets=offsets, set_counts=counts,
                    residual_full=residual_full)


def moe_workload(name, T, H, num_experts, topk, seed, *, eps=1e-6,
                 residual=True) -> Workload:
    """Deferred-finalize inputs: expert-sorted expert_out [T*topk, H], idx, w."""
    logits = _rng(seed, _S_LOGITS).standard_normal((T, num_experts), dtype=np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :topk]     # ties: lower id
    chosen = np.take_along_axis(logits, order, axis=1).astype(np.float64)
    ex = np.exp(chosen - chosen.max(axis=1, keepdims=True))
    w = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)
    experts = order.astype(np.int64)
    tok = np.repeat(np.arange(T, dtype=np.int64), topk)
    slot = np.tile(np.arange(topk, dtype=np.int64), T)
    perm = np.lexsort((slot, tok, experts.reshape(-1)))              # by expert, t, j
    idx = np.empty(T * topk, np.int32)
    idx[perm] = np.arange(T * topk, dtype=np.int32)
    expert_out = normal_bf16(seed, _S_EXPERT, (T * topk, H))
    res = normal_bf16(seed, _S_RESIDUAL, (T, H)) if residual else None
    return Workload(name=name, T=T, H=H, eps=eps, gamma=gamma_f32(seed, H),
                    residual=res, expert_out=expert_out, idx=idx.reshape(T, topk),
                    w=w, topk=topk, num_experts=num_experts)


# The five workloads the boundary is specified on (seed = position in this list).
def tiny_fold_norm(seed=0):
    """K=2 partials [16,512] ~N(0,1), residual ~N(0,1): residual' and bf16 y."""
    return fold_workload("tiny_fold_norm", 2, 16, 512, seed)


def decode_fold_norm(seed=1, initial=False):
    """K=8 partials [64,4096] ~N(0,0.5^2), residual ~N(0,1); initial=True drops the
    residual (Initial stream state: residual' = sum of partials)."""
    return fold_workload("decode_initial" if initial else "decode_fold_norm", 8, 64,
                         4096, seed, partial_std=0.5, residual=not initial)


def prefill_fold_norm_fp8(seed=2, H=4096):
    """K=4 partials [2048,4096] ~N(0,1) with 1% of rows x50, residual ~N(0,1),
    RMSNorm then per-token dynamic FP8 E4M3.  (Another H gives the same recipe at that
    hidden size, for sweeps and profiles of other widths.)"""
    return fold_workload("prefill_fold_norm_fp8", 4, 2048, H, seed,
                         outlier_frac=0.01, fp8=True)


RAGGED_COUNTS = (37, 512, 5, 1470)


def ragged_slice(seed=3, slice_=3):
    """Token sets {37,512,5,1470} padded to multiples of 8 (T_pad 2032), K=8 partials
    [2032,4096]; slice `slice_` of 8 equal slices (S = 254)."""
    return slice_workload("ragged_slice", 8, 4096, RAGGED_COUNTS, 8, slice_, seed)


def moe_finalize(seed=4):
    """T=1024 tokens, 128 experts, top-8, expert_out [8192,4096] ~N(0,1)."""
    return moe_workload("moe_finalize", 1024, 4096, 128, 8, seed)


WORKLOADS = {
    "tiny_fold_norm": tiny_fold_norm,
    "decode_fold_norm": decode_fold_norm,
    "decode_initial": lambda seed=1: decode_fold_norm(seed, initial=True),
    "prefill_fold_norm_fp8": prefill_fold_norm_fp8,
    "ragged_slice": ragged_slice,
    "moe_finalize": moe_finalize,
}
