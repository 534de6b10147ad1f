"""Seeded synthetic workloads for the MTP verify / draft-input hot path.

This module only makes inputs: logits, draft ids, per-row sampling parameters and the
draft head's activations and weights.  It holds none of the method's arithmetic (no
softmax, filtering, acceptance test or normalisation).  Draft ids for sampled rows are
drawn with the Gumbel-max trick from softmax(Q / tau), restricted to the top-k ids of Q
when top-k is on; top-p is not applied, so a draft may fall outside the filtered draft
support, which exercises the verifier's "outside the support" branch.

The five workloads follow the pages' settings (a draft head of hidden size H, D draft
positions, vocabularies of 32k-262k ids); the numbers are synthetic stand-ins for the
real model's logits and weights, which are not used.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np


# ---------------------------------------------------------------- dtype helpers

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


# ---------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Workload:
    """One synthetic verify + draft-input workload."""
    name: str
    B: int                      # rows (sequences)
    D: int                      # draft positions per row
    V: int                      # vocabulary
    H: int                      # draft head hidden size
    dtype: str = "f32"          # logits storage: "f32" or "bf16"
    mode: str = "sample"        # "greedy": every row greedy; "sample": per-row temperature
    tau: float = 1.0            # temperature of sampled rows (when tau_range is None)
    tau_range: tuple | None = None
    greedy_frac: float = 0.0    # leading fraction of rows with temperature 0
    top_k: int = 0              # 0: off
    top_p: float = 1.0          # 1.0: off
    t_std: float = 3.0          # target logits ~ N(0, t_std)
    q_noise: float = 1.0        # draft logits = target + N(0, q_noise)
    q_noise_range: tuple | None = None
    draft_hit: float = 0.6      # greedy workloads: P(draft = target argmax)
    seed: int = 0               # numpy seed of the data
    philox_seed: int = 0        # seed of the verifier's counter-based uniforms
    M: int = 0                  # tokens into the draft-input stage (0: B * D)
    draft_steps: int = 1        # sequential draft-input calls (each M tokens)
    w_std: float = 0.02         # eh_proj weight ~ N(0, w_std)
    norm_w_std: float = 0.1     # RMSNorm weights ~ 1 + N(0, norm_w_std)
    emb_std: float = 1.0        # embeddings / hidden ~ N(0, emb_std)
    eps: float = 1e-6

    @property
    def tokens(self) -> int:
        return self.M if self.M else self.B * self.D

    @property
    def n_greedy_rows(self) -> int:
        if self.mode == "greedy":
            return self.B
        return int(round(self.greedy_frac * self.B))

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # greedy MTP step: one row, one draft, fp32 logits of a 32k vocabulary
    "greedy_b1_d1_v32k": Workload(
        name="greedy_b1_d1_v32k", B=1, D=1, V=32768, H=1024, mode="greedy", t_std=2.0,
        draft_hit=0.6, seed=0, philox_seed=0, w_std=0.02),
    # sampling verify: 8 rows x 3 drafts, temperature 0.7, top-k 50, top-p 0.9
    "sample_b8_d3_v152k": Workload(
        name="sample_b8_d3_v152k", B=8, D=3, V=151936, H=2048, tau=0.7, top_k=50, top_p=0.9,
        t_std=3.0, q_noise=1.0, seed=1, philox_seed=1, w_std=0.02),
    # long draft: one row x 6 drafts, bf16 logits of a 262k vocabulary, 6 sequential
    # draft-input calls of one token each
    "sample_b1_d6_v262k_bf16": Workload(
        name="sample_b1_d6_v262k_bf16", B=1, D=6, V=262144, H=1536, dtype="bf16", tau=1.0,
        top_k=64, top_p=0.95, t_std=2.5, q_noise=0.7, seed=3, philox_seed=3, M=1,
        draft_steps=6, w_std=0.02),
    # batched serving: 256 rows x 3 drafts; the first quarter of the rows greedy, the
    # rest at temperatures U[0.5, 1.2] with top-p 0.9; 768 draft-input tokens
    "serve_b256_d3_v152k": Workload(
        name="serve_b256_d3_v152k", B=256, D=3, V=151936, H=4096, tau_range=(0.5, 1.2),
        greedy_frac=0.25, top_p=0.9, t_std=3.0, q_noise_range=(0.3, 2.0), seed=4,
        philox_seed=4, M=768, w_std=0.01),
    # large hidden size: 64 rows x 1 draft, no filtering, H = 7168
    "mtp_b64_d1_v129k_h7168": Workload(
        name="mtp_b64_d1_v129k_h7168", B=64, D=1, V=129280, H=7168, tau=1.0, t_std=3.0,
        q_noise=1.0, seed=5, philox_seed=5, w_std=0.01),
}

WORKLOAD_ORDER = list(WORKLOADS)


def _normal(rng, shape, std):
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return x if dtype == "f32" else f32_to_bf16_bits(x)


def _as_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    return x if dtype == "f32" else bf16_bits_to_f32(x)


def make_verify_inputs(w: Workload) -> dict:
    """Target logits T [B, D+1, V], draft logits Q [B, D, V], draft ids d [B, D] and the
    per-row temperature / top-k / top-p arrays of a workload."""
    rng = np.random.default_rng(w.seed)
    B, D, V = w.B, w.D, w.V
    T = _store(_normal(rng, (B, D + 1, V), w.t_std), w.dtype)
    Tf = _as_f32(T, w.dtype)
    if w.q_noise_range is not None:
        sig = rng.uniform(*w.q_noise_range, size=B).astype(np.float32)
    else:
        sig = np.full(B, w.q_noise, np.float32)
    Q = Tf[:, :D, :] + _normal(rng, (B, D, V), 1.0) * sig[:, None, None]
    Q = _store(Q.astype(np.float32), w.dtype)
    Qf = _as_f32(Q, w.dtype)

    ng = w.n_greedy_rows
    tau = np.zeros(B, np.float32)
    if w.mode != "greedy":
        if w.tau_range is not None:
            tau[ng:] = rng.uniform(*w.tau_range, size=B - ng).astype(np.float32)
        else:
            tau[ng:] = np.float32(w.tau)
    top_k = np.full(B, w.top_k, np.int32)
    top_p = np.full(B, w.top_p, np.float32)

    d = np.zeros((B, D), np.int32)
    for b in range(B):
        for j in range(D):
            if w.mode == "greedy":
                # the target's own choice with probability draft_hit, else a uniform id
                if rng.random() < w.draft_hit:
                    d[b, j] = int(np.argmax(Tf[b, j]))
                else:
                    d[b, j] = int(rng.integers(0, V))
            elif b < ng:
                d[b, j] = int(np.argmax(Qf[b, j]))  # a greedy drafter's pick
            else:
                g = -np.log(-np.log(rng.random(V)))
                score = Qf[b, j].astype(np.float64) / float(tau[b]) + g
                if w.top_k and w.top_k < V:
                    ids = np.argpartition(-Qf[b, j], w.top_k - 1)[:w.top_k]
                    d[b, j] = int(ids[np.argmax(score[ids])])
                else:
                    d[b, j] = int(np.argmax(score))
    return dict(T=T, Q=Q, d=d, tau=tau, top_k=top_k, top_p=top_p, seed=w.philox_seed,
                dtype=w.dtype, B=B, D=D, V=V)


def make_draft_input(w: Workload, seed_offset: int = 1000) -> dict:
    """Draft-head input stage: embeddings e and hidden states h [steps, M, H], the two
    RMSNorm weights [H] and the eh_proj weight W [H, 2H], all as bf16 bits."""
    rng = np.random.default_rng(w.seed + seed_offset)
    M, H, S = w.tokens, w.H, w.draft_steps
    e = f32_to_bf16_bits(_normal(rng, (S, M, H), w.emb_std))
    h = f32_to_bf16_bits(_normal(rng, (S, M, H), w.emb_std))
    we = f32_to_bf16_bits(1.0 + _normal(rng, (H,), w.norm_w_std))
    wh = f32_to_bf16_bits(1.0 + _normal(rng, (H,), w.norm_w_std))
    W = f32_to_bf16_bits(_normal(rng, (H, 2 * H), w.w_std))
    return dict(e=e, h=h, we=we, wh=wh, W=W, eps=w.eps, M=M, H=H, steps=S)


def make_greedy_draft_logits(w: Workload, rows: int | None = None) -> np.ndarray:
    """Draft logits [rows, V] for a greedy-draft call (fp32 ~ N(0, t_std), or bf16)."""
    rng = np.random.default_rng(w.seed + 2000)
    rows = w.tokens if rows is None else rows
    return _store(_normal(rng, (rows, w.V), w.t_std), w.dtype)


def make_lm_head_input(M: int, H: int, V: int, seed: int, w_std: float = 0.02,
                       hidden_std: float = 1.0, norm_w_std: float = 0.1) -> dict:
    """The draft head's output layer: hidden states [M, H] ~ N(0, hidden_std), the final
    norm weight [H] ~ 1 + N(0, norm_w_std) and the output-layer weight [V, H] ~ N(0, w_std),
    all as bf16 bits (random stand-ins for the shared lm_head)."""
    rng = np.random.default_rng(seed)
    hidden = f32_to_bf16_bits(_normal(rng, (M, H), hidden_std))
    norm_w = f32_to_bf16_bits(1.0 + _normal(rng, (H,), norm_w_std))
    W = np.empty((V, H), np.uint16)
    step = max(1, (1 << 24) // max(H, 1))  # rows per chunk: bounded temporaries
    for v0 in range(0, V, step):
        v1 = min(V, v0 + step)
        W[v0:v1] = f32_to_bf16_bits(_normal(rng, (v1 - v0, H), w_std))
    return dict(hidden=hidden, norm_w=norm_w, W=W, M=M, H=H, V=V, eps=1e-6)
