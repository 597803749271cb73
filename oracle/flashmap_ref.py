"""FlashMap one-jump block-draft step: the oracle.

TEST INFRASTRUCTURE ONLY. This module is a plain, slow, obviously correct CPU
statement of what the block-draft step computes, written in NumPy float64 from
the FlashMap pages. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import or run it; the library
(``include/flashmap.h`` and the CUDA sources) never does, and this module imports
nothing from the library. The two share no code, tables or constants.

Sources (each function cites the page and the section it follows):
  * ``flashmap/modeling_flashmap.py`` -- the transformers reference model
    (``rope_tables``, ``apply_rope``, ``FlashMapRMSNorm``, ``FlashMapTimeEmbedding``,
    ``FlashMapAdaLayerNorm``, ``FlashMapAttention``, ``FlashMapLayer``,
    ``FlashMapDraftModel.extend_context / mix_state / target_constants / draft``).
  * ``flashmap/configuration_flashmap.py`` -- ``FlashMapConfig``, ``DEFAULT_JUMP_GRIDS``.
  * ``flashmap/sglang/model.py`` -- the one-jump shortcut (``_draft_impl``), the
    all-layer context K/V weight (``load_weights``), the fold (``_fold_lm_head``),
    the anchor row (``forward``, ``_anchor_kv_impl``), the commit-masked write
    (``write_target_hidden_kv``), FP8 copies (``_quantize_fp8``).
  * ``flashmap/vllm/model.py`` -- position-keyed draft noise (module docstring,
    ``_noise``), ``seqused_k = p + 1`` (``_prologue``), the modulation table
    ``(layers, 9, dim)`` (``prepare``).
  * ``flashmap/sglang/sampler.py`` -- whole-block sampling, Gumbel-max with
    in-kernel Philox, the ``-inf`` full-vocabulary scatter (module docstring,
    ``IdentityMarkov.sample_block``, ``_FullLogits``).
  * tokenspeed ``dflash.py`` -- ``req_to_page`` / ``page_size`` slot addressing
    (``DFlash._draft_native``, ``compute_out_cache_loc_uniform``).
  * Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
    as 1, 2, 3" (SC'11), section 3 (the Philox round and key schedule).

Readings where the pages are silent (each the plainest one the rest of the pages support):
  R1 the noise of slot k of request b is keyed by (seed_b, position p_b+1+k);
  R2 Philox4x32-10 with key (seed lo32, seed hi32); counter (j/4, position,
     domain, step) with domain 0 = DiT noise (step 0), 1 = Gumbel noise;
  R3 a word w maps to U = ((w >> 9) + 1/2) * 2^-23, exact in float32, in (0, 1);
  R4 normals by Box-Muller on the word pairs (w0, w1) and (w2, w3);
  R5 Gumbel-max: token = argmax_j (l_j / T + G_j), G = -ln(-ln U); lowest index
     wins ties; T <= 0 or greedy -> argmax_j l_j;
  R6 RoPE angle = float32(float32(p) * inv_freq), inv_freq = float32(theta^(-2i/hd));
  R7 candidate c of a multi-candidate (tree) draft keys its noise with counter word
     3 = c (the single draft is candidate 0);
  R8 a several-jump draft starts from V-wide noise keyed like the one-jump noise
     (columns 0..V-1 instead of 0..H-1);
  R9 the folded-noise eigenbasis lists eigenvalues ascending, and each eigenvector's
     entry of largest magnitude (the first such) is made positive.

Pinning (what fixes each function other than itself; see tests/test_oracle_pins.py):
  philox4x32_10          published known-answer vectors (tests/golden/philox_kat.txt)
  uniform/normals/gumbel exact word->U map; moments, KS and chi-square laws
  rope                   closed-form rotation, norm, relative-position identity
  rms_norm/layer_norm/   closed forms and library routines (scipy erf / norm.cdf)
  gelu/silu/time_embed
  attention              brute-force pure-Python softmax on tiny shapes
  load_constants         L L^T = E^T E; fold identity; uniform constant closed form;
                         cov(z L^T) vs E^T E and vs direct x0 @ E draws
  slots/out_loc          brute-force page walk
  sample_rows            greedy = argmax; Gumbel-max frequencies vs softmax(l/T);
                         row independence; -inf outside the draft vocabulary
  noise_basis            closed-form 2 x 2 eigenpairs; Q diag(lam) Q^T = E^T E,
                         Q^T Q = I; ascending; the sign rule
  folded_noise           the fold identity against the unfolded rms_norm / x_embed;
                         cov of z diag(sqrt lam) Q^T against E^T E
  adaln / time_cond     distinct bias chunks come back as (1 + scale, shift, gate)
                         per norm and branch; time_embed reads s, jump_embed t
  dit_layer              each branch isolated by zero gates against scipy z-score /
                         norm.cdf and the pinned primitives (MLP scale/shift/gate,
                         cross-attention over one position, uniform non-causal
                         self-attention); slot permutation equivariance
  draft_request          slots at anchor + 1 + k (constant-query case); invariance
                         to shifting every position at noise_scale 0; zero gates
                         give the plain LayerNorm of the embedding
  quantize_query_e4m3    a hand-worked per-head case (ties, the 1e-12 floor)
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
from scipy.special import erf

# ---------------------------------------------------------------------------------
# Configuration and constants printed on the pages
# ---------------------------------------------------------------------------------

# configuration_flashmap.py, DEFAULT_JUMP_GRIDS: jump times per number of steps,
# endpoints exactly 0 and 1. The one-jump step uses grid "1".
DEFAULT_JUMP_GRIDS = {
    "1": [0.0, 1.0],
    "2": [0.0, 0.8172569274902344, 1.0],
    "3": [0.0, 0.8010796308517456, 0.8310279846191406, 1.0],
    "4": [0.0, 0.7906050682067871, 0.8172569274902344, 0.8379518389701843, 1.0],
}


@dataclass
class Config:
    """FlashMapConfig (configuration_flashmap.py) restricted to the fields the
    one-jump draft step reads, plus the paging of the draft KV pool."""

    target_hidden: int
    num_target_layers: int
    hidden: int
    num_layers: int
    num_heads: int
    head_dim: int
    intermediate: int
    cond_dim: int
    time_embed_dim: int
    block_size: int
    vocab_size: int
    draft_vocab_size: int
    page_size: int
    rope_theta: float = 1e4
    time_scale: float = 1000.0
    rms_norm_eps: float = 1e-6
    qk_norm_eps: float = 1e-5
    layer_norm_eps: float = 1e-6
    noise_gate_constant: bool = False  # False: "jump" gate, True: "constant"
    num_steps: int = 1
    kv_dtype: str = ""  # "e4m3": the draft KV pool stores e4m3 keys/values (else act dtype)
    noise_path: int = 0  # 0: the noise read as z L^T; 1: the folded eigenbasis (one jump)

    @staticmethod
    def from_dict(d: dict) -> "Config":
        names = Config.__dataclass_fields__.keys()
        return Config(**{k: d[k] for k in names if k in d})


# ---------------------------------------------------------------------------------
# Philox4x32-10 and the noise built from it (Salmon et al., SC'11, section 3)
# ---------------------------------------------------------------------------------

_MASK32 = np.uint64(0xFFFFFFFF)
# The Philox4x32 round multipliers and the Weyl key increments of the paper.
_PHILOX_M0 = np.uint64(0xD2511F53)
_PHILOX_M1 = np.uint64(0xCD9E8D57)
_PHILOX_W0 = np.uint64(0x9E3779B9)
_PHILOX_W1 = np.uint64(0xBB67AE85)


def philox4x32_10(counters, keys) -> np.ndarray:
    """Philox4x32 with 10 rounds (Salmon et al., section 3).

    counters: (n, 4) uint32 words (c0, c1, c2, c3); keys: (n, 2) uint32 (k0, k1).
    A round multiplies c0 and c2 by the two multipliers into 64-bit products
    (hi, lo) and outputs (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0); the key is
    bumped by the Weyl constants between rounds. Returns (n, 4) uint32."""
    c = np.asarray(counters, dtype=np.uint64).reshape(-1, 4).copy()
    k = np.asarray(keys, dtype=np.uint64).reshape(-1, 2).copy()
    c0, c1, c2, c3 = c[:, 0], c[:, 1], c[:, 2], c[:, 3]
    k0, k1 = k[:, 0], k[:, 1]
    for r in range(10):
        if r:
            k0 = (k0 + _PHILOX_W0) & _MASK32
            k1 = (k1 + _PHILOX_W1) & _MASK32
        p0 = _PHILOX_M0 * c0  # < 2^64: exact in uint64
        p1 = _PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=1).astype(np.uint32)


def seed_key(seed: int) -> tuple[int, int]:
    """Reading R2: the Philox key of a request's 64-bit seed (lo32, hi32)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & 0xFFFFFFFF, seed >> 32


def word_to_uniform(w) -> np.ndarray:
    """Reading R3: U = ((w >> 9) + 1/2) * 2^-23, in (0, 1); every value is exact
    in float32 (23 significant bits plus the half)."""
    w = np.asarray(w, dtype=np.uint64)
    return ((w >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0**-23


def box_muller(wa, wb) -> tuple[np.ndarray, np.ndarray]:
    """Reading R4: two standard normals from two words (textbook Box-Muller)."""
    ua, ub = word_to_uniform(wa), word_to_uniform(wb)
    r = np.sqrt(-2.0 * np.log(ua))
    return r * np.cos(2.0 * np.pi * ub), r * np.sin(2.0 * np.pi * ub)


def _philox_rows(seed: int, positions, ncols: int, domain: int, step: int) -> np.ndarray:
    """Words for columns 0..ncols-1 of rows keyed by ``positions``: counter
    (j/4, position, domain, step), word j mod 4 (reading R2).
    Returns (len(positions), ceil(ncols/4), 4) uint32."""
    pos = np.atleast_1d(np.asarray(positions, dtype=np.int64))
    n4 = (ncols + 3) // 4
    ctr = np.zeros((len(pos), n4, 4), dtype=np.uint64)
    ctr[:, :, 0] = np.arange(n4, dtype=np.uint64)[None, :]
    ctr[:, :, 1] = (pos.astype(np.uint64) & _MASK32)[:, None]
    ctr[:, :, 2] = np.uint64(domain)
    ctr[:, :, 3] = np.uint64(step & 0xFFFFFFFF)
    k0, k1 = seed_key(seed)
    keys = np.empty((len(pos) * n4, 2), dtype=np.uint64)
    keys[:, 0], keys[:, 1] = k0, k1
    return philox4x32_10(ctr.reshape(-1, 4), keys).reshape(len(pos), n4, 4)


def draft_normals(seed: int, positions, ncols: int, candidate: int = 0) -> np.ndarray:
    """The starting noise z ~ N(0, I_H) of each slot (flashmap/vllm/model.py,
    module docstring: noise keyed by the request's seed and the slot's position;
    readings R1, R2, R4). Row i is keyed by positions[i]; returns (len, ncols):
    column j is normal j mod 4 of counter j/4, the normals of a counter being the
    Box-Muller pairs of its words (w0, w1) and (w2, w3). Candidate c of a
    multi-candidate (tree) draft takes counter word 3 = c (reading R7), so candidate
    0 is the single draft."""
    w = _philox_rows(seed, positions, ncols, domain=0, step=candidate)
    n0, n1 = box_muller(w[..., 0], w[..., 1])
    n2, n3 = box_muller(w[..., 2], w[..., 3])
    out = np.stack([n0, n1, n2, n3], axis=-1).reshape(w.shape[0], -1)
    return out[:, :ncols]


def gumbel_noise(seed: int, position: int, step: int, ncols: int) -> np.ndarray:
    """Gumbel noise G = -ln(-ln U) for one block row (flashmap/sglang/sampler.py,
    module docstring: Gumbel-max with in-kernel Philox noise; readings R2, R3, R5)."""
    w = _philox_rows(seed, [int(position)], ncols, domain=1, step=step).reshape(-1)[:ncols]
    return -np.log(-np.log(word_to_uniform(w)))


# ---------------------------------------------------------------------------------
# Elementwise and row operations (modeling_flashmap.py)
# ---------------------------------------------------------------------------------


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """modeling_flashmap.py, rope_tables: inv_freq_i = theta^(-2i/hd), in float32
    (reading R6: computed in float64, rounded once to float32)."""
    i = np.arange(0, head_dim, 2, dtype=np.float64)
    return (1.0 / theta ** (i / head_dim)).astype(np.float32)


def rope_angles(positions, head_dim: int, theta: float) -> np.ndarray:
    """modeling_flashmap.py, rope_tables: the float32 angles p * inv_freq
    (one float32-rounded product per angle). Returns (n, hd/2) float32."""
    p = np.asarray(positions, dtype=np.float32).reshape(-1, 1)
    return p * rope_inv_freq(head_dim, theta)[None, :]  # float32 * float32 -> float32


def apply_rope(x: np.ndarray, positions, theta: float) -> np.ndarray:
    """modeling_flashmap.py, apply_rope: rotate the interleaved channel pairs
    (x[2i], x[2i+1]) of x (n, heads, hd) by the angle of position n and pair i."""
    hd = x.shape[-1]
    ang = rope_angles(positions, hd, theta).astype(np.float64)  # (n, hd/2)
    cos, sin = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x, dtype=np.float64)
    out[..., 0::2] = x1 * cos - x2 * sin
    out[..., 1::2] = x2 * cos + x1 * sin
    return out


def rms_norm(x: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """modeling_flashmap.py, FlashMapRMSNorm: x * (w * rsqrt(mean(x^2) + eps)) over
    the last axis (the dtype rounding of the scale is a no-op in float64)."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x * (np.asarray(weight, dtype=np.float64) / np.sqrt(ms + eps))


def layer_norm(x: np.ndarray, eps: float) -> np.ndarray:
    """modeling_flashmap.py, FlashMapAdaLayerNorm: F.layer_norm with no affine:
    (x - mean) / sqrt(biased var + eps) over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    mu = np.mean(x, axis=-1, keepdims=True)
    var = np.mean((x - mu) ** 2, axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def gelu(x: np.ndarray) -> np.ndarray:
    """modeling_flashmap.py, FlashMapMLP: F.gelu (exact erf form)."""
    return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def time_embedding(t: float, l1_w, l1_b, l2_w, l2_b, time_embed_dim: int, time_scale: float):
    """modeling_flashmap.py, FlashMapTimeEmbedding: sinusoidal features of
    t * time_scale with freqs exp(-ln(1e4) i / half), [cos, sin], then
    linear_1 -> SiLU -> linear_2."""
    half = time_embed_dim // 2
    freqs = np.exp(-math.log(10000.0) * np.arange(half, dtype=np.float64) / half)
    args = (t * time_scale) * freqs
    emb = np.concatenate([np.cos(args), np.sin(args)])
    h = silu(_f64(l1_w) @ emb + _f64(l1_b))
    return _f64(l2_w) @ h + _f64(l2_b)


def adaln_modulation(cond, w, b):
    """modeling_flashmap.py, FlashMapAdaLayerNorm.modulation: linear(SiLU(cond))
    chunked into (scale, shift, gate)."""
    out = _f64(w) @ silu(cond) + _f64(b)
    d = out.shape[0] // 3
    return out[:d], out[d : 2 * d], out[2 * d :]


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Non-causal softmax attention per head (F.scaled_dot_product_attention with
    scale hd^-1/2). q (nq, heads, hd), k/v (nk, heads, hd) -> (nq, heads, hd)."""
    hd = q.shape[-1]
    s = np.einsum("qhd,khd->hqk", q, k) / math.sqrt(hd)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=-1, keepdims=True)
    return np.einsum("hqk,khd->qhd", p, v)


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------------
# Load-time constants
# ---------------------------------------------------------------------------------


@dataclass
class Constants:
    mods: np.ndarray  # (L, 9, D): (1+scale, shift, gate) x (self, cross, mlp)
    final: np.ndarray  # (2, D): (1+scale, shift) of the final AdaLN
    gate: float  # noise gate of the jump 0 -> 1
    uniform: np.ndarray  # (H,): state_norm(mean row of E)
    gram: np.ndarray  # (H, H) E^T E
    chol: np.ndarray  # (H, H) lower L with L L^T = E^T E
    hot: np.ndarray  # (Vd,) int64 sorted draft-vocabulary token ids
    head_w: np.ndarray  # (Vd, D) folded head
    head_b: np.ndarray  # (Vd,)
    extra: dict = field(default_factory=dict)


def jump_conditioning(cfg: Config, W: dict, s: float, t: float):
    """modeling_flashmap.py, FlashMapDraftModel.time_conditioning:
    cond = time_embed(s) + jump_embed(t); every AdaLN's (scale, shift, gate)."""
    te = lambda name, x: time_embedding(  # noqa: E731
        x, W[f"{name}.linear_1.weight"], W[f"{name}.linear_1.bias"],
        W[f"{name}.linear_2.weight"], W[f"{name}.linear_2.bias"],
        cfg.time_embed_dim, cfg.time_scale)
    cond = te("time_embed", s) + te("jump_embed", t)
    mods = np.zeros((cfg.num_layers, 9, cfg.hidden))
    for l in range(cfg.num_layers):
        for j, norm in enumerate(("self_attn_adaln", "cross_attn_adaln", "mlp_adaln")):
            sc, sh, g = adaln_modulation(cond, W[f"layers.{l}.{norm}.linear.weight"],
                                         W[f"layers.{l}.{norm}.linear.bias"])
            # flashmap/vllm/model.py, prepare: stored as (1 + scale, shift, gate).
            mods[l, 3 * j], mods[l, 3 * j + 1], mods[l, 3 * j + 2] = 1.0 + sc, sh, g
    sc, sh, _ = adaln_modulation(cond, W["final_adaln.linear.weight"], W["final_adaln.linear.bias"])
    return mods, np.stack([1.0 + sc, sh]), cond


def draft_vocabulary(cfg: Config, ranking) -> np.ndarray:
    """flashmap/sglang/model.py, prepare: hot ids = sort(ranking[:Vd]); a size
    outside (0, V) (or no ranking) means the full vocabulary."""
    vd, v = cfg.draft_vocab_size, cfg.vocab_size
    if ranking is None or not (0 < vd < v):
        return np.arange(v, dtype=np.int64)
    return np.sort(np.asarray(ranking, dtype=np.int64)[:vd])


def load_constants(cfg: Config, W: dict, E, LM, ranking, *, skip_gram: bool = False) -> Constants:
    """Everything a one-jump draft reads that depends only on the weights:
    modulations (modeling_flashmap.py, time_conditioning; flashmap/vllm/model.py,
    prepare), the uniform-posterior constant and the Cholesky factor of E^T E
    (modeling_flashmap.py, target_constants; flashmap/sglang/model.py,
    _jump_constants / _embedding_gram), the draft vocabulary and the folded head
    (flashmap/sglang/model.py, _fold_lm_head).

    skip_gram=True replaces the gram and its factor by the identity: only for
    timing runs, where the values of L do not change the work."""
    s, t = DEFAULT_JUMP_GRIDS["1"]
    mods, final, _ = jump_conditioning(cfg, W, s, t)
    # modeling_flashmap.py, mix_state: noise_gate times the jump (t - s), or alone.
    jump = 1.0 if cfg.noise_gate_constant else (t - s)
    gate = float(np.asarray(W["noise_gate"], dtype=np.float64).reshape(-1)[0]) * jump
    E64 = _f64(E)
    # The uniform posterior (1/V each) embeds to the mean row of E, then state_norm.
    uniform = rms_norm(E64.mean(axis=0), W["state_norm.weight"], cfg.rms_norm_eps)
    H = E64.shape[1]
    if skip_gram:
        gram, chol = np.eye(H), np.eye(H)
    else:
        gram = E64.T @ E64
        chol = np.linalg.cholesky(gram)  # lower, positive diagonal (unique)
    hot = draft_vocabulary(cfg, ranking)
    lm_hot = _f64(LM)[hot]
    head_w = lm_hot @ _f64(W["head.weight"])  # (Vd, H) @ (H, D)
    head_b = lm_hot @ _f64(W["head.bias"])
    C = Constants(mods=mods, final=final, gate=gate, uniform=uniform, gram=gram,
                  chol=chol, hot=hot, head_w=head_w, head_b=head_b)
    if cfg.noise_path == 1:
        C.extra["folded"] = folded_noise(cfg, W, C)
    return C


def noise_basis(gram: np.ndarray):
    """flashmap/sglang/model.py, noise_basis: (lam, Q) in float64 with
    E^T E = Q diag(lam) Q^T, lam clamped at 0. Reading R9 fixes what the pages leave to
    the eigensolver: lam ascending, and each column of Q signed so that its entry of
    largest magnitude (the first such) is positive."""
    lam, Q = np.linalg.eigh(np.asarray(gram, dtype=np.float64))
    order = np.argsort(lam, kind="stable")
    lam, Q = lam[order], Q[:, order]
    lead = np.argmax(np.abs(Q), axis=0)  # first index of the largest magnitude
    sign = np.where(Q[lead, np.arange(Q.shape[1])] < 0, -1.0, 1.0)
    return np.clip(lam, 0.0, None), Q * sign


@dataclass
class FoldedNoise:
    variance: np.ndarray  # (H,) lam / H
    proj: np.ndarray  # (H, D) M = diag(sqrt lam) Q^T diag(w) W_x^T
    embedded_uniform: np.ndarray  # (D,) x_embed(u)


def folded_noise(cfg: Config, W: dict, C: Constants) -> FoldedNoise:
    """flashmap/sglang/model.py, _folded_noise: with y = (z * sqrt(lam)) @ Q^T,
    x_embed(u + gate * noise_norm(y)) = x_embed(u) + gate * r * (z @ M),
    r = rsqrt(sum(lam z^2) / H + eps), M = diag(sqrt(lam)) Q^T diag(w) W_x^T,
    w the noise norm's weight."""
    lam, Q = noise_basis(C.gram)
    H = lam.shape[0]
    w = _f64(W["noise_norm.weight"])
    proj = (np.sqrt(lam)[:, None] * Q.T) * w[None, :] @ _f64(W["x_embed.weight"]).T
    xu = C.uniform @ _f64(W["x_embed.weight"]).T + _f64(W["x_embed.bias"])
    return FoldedNoise(variance=lam / H, proj=proj, embedded_uniform=xu)


def embed_noise_folded(cfg: Config, F: FoldedNoise, gate: float, z: np.ndarray) -> np.ndarray:
    """The x_embed output of one jump from noise z (rows, H) by the folded path
    (flashmap/vllm/model.py, _one_jump): x_embed(u) + gate * r * (z @ M)."""
    z = np.asarray(z, dtype=np.float64)
    r = 1.0 / np.sqrt((z * z) @ F.variance + cfg.rms_norm_eps)
    return F.embedded_uniform + (gate * r)[:, None] * (z @ F.proj)


# ---------------------------------------------------------------------------------
# Context keys and values (the write and the anchor row)
# ---------------------------------------------------------------------------------


def _heads(x: np.ndarray, cfg: Config) -> np.ndarray:
    return x.reshape(x.shape[0], cfg.num_heads, cfg.head_dim)


def context_kv(cfg: Config, W: dict, ctx: np.ndarray, positions) -> tuple[np.ndarray, np.ndarray]:
    """modeling_flashmap.py, FlashMapAttention.project_kv of every layer's
    cross-attention: k = RoPE(k_norm(heads(k_proj ctx))), v = heads(v_proj ctx).
    ctx (n, D) -> keys, values (L, n, heads, hd)."""
    n = ctx.shape[0]
    K = np.empty((cfg.num_layers, n, cfg.num_heads, cfg.head_dim))
    V = np.empty_like(K)
    for l in range(cfg.num_layers):
        pre = f"layers.{l}.cross_attn"
        k = _heads(ctx @ _f64(W[f"{pre}.k_proj.weight"]).T, cfg)
        k = rms_norm(k, W[f"{pre}.k_norm.weight"], cfg.qk_norm_eps)
        K[l] = apply_rope(k, positions, cfg.rope_theta)
        V[l] = _heads(ctx @ _f64(W[f"{pre}.v_proj.weight"]).T, cfg)
    return K, V


def write_rows_kv(cfg: Config, W: dict, target_hidden: np.ndarray, positions):
    """modeling_flashmap.py, extend_context (flashmap/sglang/model.py,
    _write_context): ctx = hidden_norm(fc(target hidden)), then every layer's
    context keys and values. target_hidden (n, Lt*H) -> (L, n, heads, hd) x 2."""
    ctx = rms_norm(_f64(target_hidden) @ _f64(W["fc.weight"]).T, W["hidden_norm.weight"],
                   cfg.rms_norm_eps)
    return context_kv(cfg, W, ctx, positions)


def anchor_kv(cfg: Config, W: dict, E, anchor_ids, positions):
    """modeling_flashmap.py, draft (flashmap/sglang/model.py, _anchor_kv_impl):
    the anchor's context row anchor_norm(anchor_proj(E[anchor])) projected by every
    layer's cross-attention at the anchor's position."""
    e = _f64(E)[np.asarray(anchor_ids, dtype=np.int64)]
    a = rms_norm(e @ _f64(W["anchor_proj.weight"]).T + _f64(W["anchor_proj.bias"]),
                 W["anchor_norm.weight"], cfg.rms_norm_eps)
    return context_kv(cfg, W, a, positions)


def slot_of(req_to_page: np.ndarray, req: int, pos: int, page_size: int) -> int:
    """tokenspeed dflash.py, DFlash._draft_native (compute_out_cache_loc_uniform):
    loc = req_to_page[req, pos / page] * page + pos % page."""
    return int(req_to_page[req, pos // page_size]) * page_size + pos % page_size


def write_locations(start_pos, commit_lens, window: int, req_pool_idx, req_to_page, page_size):
    """flashmap/sglang/model.py, write_target_hidden_kv (verify windows): column c of
    request b sits at position start_pos[b] + c and is written only if
    c < commit_lens[b] (all columns without commit_lens). Returns (bs, W) int64
    slots, -1 where skipped."""
    bs = len(start_pos)
    out = np.full((bs, window), -1, dtype=np.int64)
    for b in range(bs):
        n = window if commit_lens is None else int(commit_lens[b])
        for c in range(min(n, window)):
            out[b, c] = slot_of(req_to_page, int(req_pool_idx[b]), int(start_pos[b]) + c, page_size)
    return out


# ---------------------------------------------------------------------------------
# The one-jump draft of one request
# ---------------------------------------------------------------------------------


def embed_noise(cfg: Config, W: dict, C: Constants, z: np.ndarray) -> np.ndarray:
    """The one-jump state embedding from z ~ N(0, I_H): u + gate * noise_norm(z L^T)
    (modeling_flashmap.py, mix_state at s = 0, the noise read as z L^T)."""
    return C.uniform + C.gate * rms_norm(z @ C.chol.T, W["noise_norm.weight"], cfg.rms_norm_eps)


def noise_embedding(cfg: Config, W: dict, C: Constants, seed: int, positions, noise_scale: float,
                    candidate: int = 0):
    """flashmap/sglang/model.py, _draft_impl (one jump from t = 0): the embedded
    state u + gate * noise_norm(z L^T) with z keyed by the slot positions (and the
    candidate), then x_embed. Returns (K, D)."""
    z = noise_scale * draft_normals(seed, positions, cfg.target_hidden, candidate)
    if cfg.noise_path == 1:  # the folded eigenbasis (flashmap/sglang/model.py, _folded_noise)
        return embed_noise_folded(cfg, C.extra["folded"], C.gate, z)
    e = embed_noise(cfg, W, C, z)
    return e @ _f64(W["x_embed.weight"]).T + _f64(W["x_embed.bias"])


def _linear(x: np.ndarray, w) -> np.ndarray:
    return x @ _f64(w).T


def dit_layer(cfg: Config, W: dict, l: int, mods: np.ndarray, x: np.ndarray, positions,
              contexts) -> np.ndarray:
    """modeling_flashmap.py, FlashMapLayer.forward on the blocks of one or more requests,
    x (n_req * K, D), row i * K + k being slot k of request i at positions[i*K + k]:
    self-attention across each request's own K slots, cross-attention onto that
    request's context contexts[i] = (keys, values) (n_i, heads, hd) (positions 0..p_i),
    MLP; each behind a modulated LayerNorm and a gated residual. Requests never mix:
    every linear acts row by row, every attention within one request."""
    eps = cfg.layer_norm_eps
    K = cfg.block_size
    pre = f"layers.{l}"
    m = mods
    nreq = x.shape[0] // K
    # self-attention
    h = layer_norm(x, eps) * m[0] + m[1]
    sa = f"{pre}.self_attn"
    q = rms_norm(_heads(_linear(h, W[f"{sa}.q_proj.weight"]), cfg), W[f"{sa}.q_norm.weight"], cfg.qk_norm_eps)
    k = rms_norm(_heads(_linear(h, W[f"{sa}.k_proj.weight"]), cfg), W[f"{sa}.k_norm.weight"], cfg.qk_norm_eps)
    v = _heads(_linear(h, W[f"{sa}.v_proj.weight"]), cfg)
    q, k = apply_rope(q, positions, cfg.rope_theta), apply_rope(k, positions, cfg.rope_theta)
    att = np.concatenate([attention(q[i * K:(i + 1) * K], k[i * K:(i + 1) * K], v[i * K:(i + 1) * K])
                          for i in range(nreq)]).reshape(x.shape[0], -1)
    x = x + m[2] * _linear(att, W[f"{sa}.o_proj.weight"])
    # cross-attention
    h = layer_norm(x, eps) * m[3] + m[4]
    ca = f"{pre}.cross_attn"
    q = rms_norm(_heads(_linear(h, W[f"{ca}.q_proj.weight"]), cfg), W[f"{ca}.q_norm.weight"], cfg.qk_norm_eps)
    q = apply_rope(q, positions, cfg.rope_theta)
    qs = [q[i * K:(i + 1) * K] for i in range(nreq)]
    if cfg.kv_dtype == "e4m3":  # e4m3 pool: the queries are quantized per (request, head)
        qs = [quantize_query_e4m3(qi) for qi in qs]
    ctx = np.concatenate([attention(qs[i], contexts[i][0], contexts[i][1])
                          for i in range(nreq)]).reshape(x.shape[0], -1)
    x = x + m[5] * _linear(ctx, W[f"{ca}.o_proj.weight"])
    # MLP
    h = layer_norm(x, eps) * m[6] + m[7]
    f1 = gelu(_linear(h, W[f"{pre}.mlp.fc1.weight"]) + _f64(W[f"{pre}.mlp.fc1.bias"]))
    x = x + m[8] * (_linear(f1, W[f"{pre}.mlp.fc2.weight"]) + _f64(W[f"{pre}.mlp.fc2.bias"]))
    return x


def draft_requests(cfg: Config, W: dict, C: Constants, ctx_kv: list, anchor_pos: list, seeds: list,
                   noise_scale: float = 1.0, candidates: list | None = None) -> np.ndarray:
    """modeling_flashmap.py, FlashMapDraftModel.draft with one step, for requests i whose
    cross-attention context (anchor included) is ctx_kv[i] = (keys, values), each
    (L, p_i + 1, heads, hd): slots at positions p_i+1 .. p_i+K; returns the final AdaLN
    output (n_req, K, D), which the folded head maps to logits. A tree draft's
    candidate blocks are entries with the same context, position and seed and their
    own candidate index (flashmap/sglang/model.py, _draft_impl with n_cand > 1: the
    same blocks from independent noise)."""
    K = cfg.block_size
    nreq = len(anchor_pos)
    candidates = candidates if candidates is not None else [0] * nreq
    positions = np.concatenate([p + 1 + np.arange(K) for p in anchor_pos])
    for (kc, _), p in zip(ctx_kv, anchor_pos):
        assert kc.shape[1] == p + 1, "context is positions 0..p"
    x = np.concatenate([noise_embedding(cfg, W, C, s, p + 1 + np.arange(K), noise_scale, c)
                        for s, p, c in zip(seeds, anchor_pos, candidates)])
    for l in range(cfg.num_layers):
        x = dit_layer(cfg, W, l, C.mods[l], x, positions, [(kc[l], vc[l]) for kc, vc in ctx_kv])
    out = layer_norm(x, cfg.layer_norm_eps) * C.final[0] + C.final[1]
    return out.reshape(nreq, K, -1)


def draft_request(cfg: Config, W: dict, C: Constants, ctx_k: np.ndarray, ctx_v: np.ndarray,
                  anchor_pos: int, seed: int, noise_scale: float = 1.0) -> np.ndarray:
    """draft_requests for a single request: (K, D)."""
    return draft_requests(cfg, W, C, [(ctx_k, ctx_v)], [anchor_pos], [seed], noise_scale)[0]


def head_logits(C: Constants, hidden: np.ndarray) -> np.ndarray:
    """flashmap/sglang/model.py, head_logits: the folded head over the draft
    vocabulary, (rows, D) -> (rows, Vd)."""
    return _f64(hidden) @ C.head_w.T + C.head_b


# ---------------------------------------------------------------------------------
# Whole-block sampling
# ---------------------------------------------------------------------------------


def sample_rows(logits: np.ndarray, temperature, greedy, seeds, positions, step: int, hot):
    """flashmap/sglang/sampler.py, FlashMapDraftSampler.__call__ (fused variant):
    every row of the block at once; greedy rows (or T <= 0) take argmax_j l_j,
    the others argmax_j (l_j / T + G_j) with G from the row's Philox stream
    (readings R2, R3, R5); drafted index j -> token hot[j].

    The decision is taken in float32 (the logits are rounded to float32 first),
    as the library takes it. Returns (tokens int64 (rows,), index (rows,),
    top-2 margin of the maximised quantity (rows,))."""
    lg = np.asarray(logits, dtype=np.float64)
    rows = lg.shape[0]
    tokens = np.empty(rows, dtype=np.int64)
    index = np.empty(rows, dtype=np.int64)
    margin = np.empty(rows, dtype=np.float64)
    for r in range(rows):
        l32 = lg[r].astype(np.float32)
        t = float(temperature[r])
        if bool(greedy[r]) or t <= 0.0:
            val = l32
        else:
            g = gumbel_noise(int(seeds[r]), int(positions[r]), step, lg.shape[1]).astype(np.float32)
            val = (l32 / np.float32(t)).astype(np.float32) + g
        j = int(np.argmax(val))  # first maximum: lowest index wins ties
        index[r], tokens[r] = j, int(hot[j])
        srt = np.sort(val.astype(np.float64))
        margin[r] = srt[-1] - srt[-2] if len(srt) > 1 else np.inf
    return tokens, index, margin


def full_logits(logits: np.ndarray, hot, vocab_size: int) -> np.ndarray:
    """flashmap/sglang/sampler.py, IdentityMarkov.sample_block / _FullLogits: the
    draft-vocabulary logits scattered over the full vocabulary, -inf elsewhere."""
    out = np.full((logits.shape[0], vocab_size), -np.inf)
    out[:, np.asarray(hot)] = logits
    return out


# ---------------------------------------------------------------------------------
# FP8 (e4m3) weight copies, per output channel
# ---------------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_round(x) -> np.ndarray:
    """Round float32 values to the nearest e4m3fn value (ties to even),
    saturating at +-448: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
    subnormal step 2^-9. Returns float64 holding exact e4m3 values."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # exponent of the e4m3 binade of a (normals have e >= -6; below, step 2^-9)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))  # a = m 2^ex, m in [1/2, 1)
    e = np.maximum(ex.astype(np.float64) - 1.0, -6.0)
    step = 2.0 ** (e - 3)
    q = np.round(a / step) * step  # np.round: ties to even; a/step exact (powers of 2)
    q = np.minimum(q, E4M3_MAX)
    return np.sign(x) * q


def quantize_e4m3_per_channel(w) -> tuple[np.ndarray, np.ndarray]:
    """flashmap/sglang/model.py, _quantize_fp8 (quantize_weight_fp8): per output
    channel scale = max|w_row| / 448 in float32 (an all-zero row gets 1) and
    q = e4m3(w / scale) with the division in float32. Returns (q, scale) with q
    the exact e4m3 values (float64) and scale float32 (rows,)."""
    w32 = np.asarray(w, dtype=np.float32)
    amax = np.max(np.abs(w32), axis=1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    scale = np.where(amax > 0, scale, np.float32(1.0)).astype(np.float32)
    q = e4m3_round((w32 / scale[:, None]).astype(np.float32))
    return q, scale


def dequantize(q: np.ndarray, scale: np.ndarray) -> np.ndarray:
    return _f64(q) * _f64(scale)[:, None]


def e4m3_linear_names(cfg: Config) -> list:
    """flashmap/sglang/model.py, _quantize_fp8: the weights with e4m3 copies, by their
    module names: x_embed, fc, anchor_proj, every block's self q/k/v (the fused qkv)
    and o, cross q and o, the cross k/v (the all-layer context K/V weight), fc1 and
    fc2. The folded head is quantized too (e4m3_constants); the noise factor L, the
    norms and the AdaLN weights stay in the activation dtype."""
    names = ["x_embed.weight", "fc.weight", "anchor_proj.weight"]
    for l in range(cfg.num_layers):
        p = f"layers.{l}"
        names += [f"{p}.self_attn.{x}_proj.weight" for x in ("q", "k", "v", "o")]
        names += [f"{p}.cross_attn.{x}_proj.weight" for x in ("q", "k", "v", "o")]
        names += [f"{p}.mlp.fc1.weight", f"{p}.mlp.fc2.weight"]
    return names


def e4m3_weights(cfg: Config, W: dict) -> dict:
    """The weights an e4m3 drafter computes with: each quantized weight replaced by
    its dequantized copy q * scale (per output channel). Quantizing q, k and v (or
    each layer's cross k and v) separately equals quantizing their row concatenation,
    as the scales are per row."""
    out = dict(W)
    for name in e4m3_linear_names(cfg):
        out[name] = dequantize(*quantize_e4m3_per_channel(W[name]))
    return out


def e4m3_constants(consts: Constants) -> Constants:
    """The folded head of an e4m3 drafter: W_f quantized per output channel after
    folding (flashmap/sglang/model.py, _quantize_fp8, "head": the folded head)."""
    from dataclasses import replace

    return replace(consts, head_w=dequantize(*quantize_e4m3_per_channel(consts.head_w)))


# ---------------------------------------------------------------------------------
# e4m3 draft KV pool (flashmap/sglang/model.py, _paged_cross_attention_fp8)
# ---------------------------------------------------------------------------------


def store_kv(cfg: Config, k: np.ndarray, v: np.ndarray) -> tuple:
    """The values a pool of cfg's kv dtype holds for keys/values k, v: e4m3 with scale
    1 (nearest even, saturated at +-448) for an e4m3 pool, else k, v themselves."""
    if cfg.kv_dtype != "e4m3":
        return k, v
    return e4m3_round(np.asarray(k, dtype=np.float32)), e4m3_round(np.asarray(v, dtype=np.float32))


def quantize_query_e4m3(q: np.ndarray) -> np.ndarray:
    """One request's queries (slots, heads, hd) as the fp8 cross-attention sees them:
    per head, scale = max(max|q| over slots and channels, 1e-12) / 448 in float32,
    q8 = e4m3(q / scale) with the division in float32; returns q8 * scale (float64),
    so that attention(q8 * scale, K, V) equals the descaled fp8 product."""
    q32 = np.asarray(q, dtype=np.float32)
    amax = np.max(np.abs(q32), axis=(0, 2))
    scale = (np.maximum(amax, np.float32(1e-12)) / np.float32(E4M3_MAX)).astype(np.float32)
    q8 = e4m3_round((q32 / scale[None, :, None]).astype(np.float32))
    return q8 * _f64(scale)[None, :, None]


# ---------------------------------------------------------------------------------
# Tree drafting: the verify tree of N candidate blocks per request
# (flashmap/sglang/tree.py, build_tree_abi)
# ---------------------------------------------------------------------------------


def build_tree(candidates, width: int):
    """The verify tree of one request's candidate blocks, stated as a trie.

    candidates (N, K) token ids drafted after the anchor (the tree's root). Every
    distinct prefix c[:d+1] of a candidate is a node at depth d; its vote is how many
    candidates share that prefix, its representative the lowest candidate index
    having it. The width - 1 nodes ranked first by (more votes, shallower, lower
    representative) are kept -- a node's parent always ranks before it -- and listed
    by (depth, representative), numbered 1.. in that order (the root is 0). With fewer
    nodes than width - 1, the list is padded with copies of the first listed node (a
    depth-0 node, parent the root).

    Returns (tokens (width-1,), ids (width-1,) = parent * width + number,
    stats (2,) = (nodes in the trie, distinct candidates))."""
    c = [tuple(int(t) for t in row) for row in np.asarray(candidates)]
    n, k = len(c), len(c[0])
    m = width - 1
    nodes = {}  # prefix -> [votes, representative]
    for i, row in enumerate(c):
        for d in range(k):
            pre = row[:d + 1]
            if pre in nodes:
                nodes[pre][0] += 1
            else:
                nodes[pre] = [1, i]
    ranked = sorted(nodes, key=lambda p: (-nodes[p][0], len(p), nodes[p][1]))
    kept = sorted(ranked[:m], key=lambda p: (len(p), nodes[p][1]))
    number = {p: q + 1 for q, p in enumerate(kept)}
    tokens, ids = [], []
    for q, p in enumerate(kept):
        parent = number[p[:-1]] if len(p) > 1 else 0
        tokens.append(p[-1])
        ids.append(parent * width + q + 1)
    for q in range(len(kept), m):  # padding: copies of the first node under the root
        tokens.append(kept[0][-1])
        ids.append(0 * width + q + 1)
    distinct = len(set(c))
    return (np.array(tokens, dtype=np.int64), np.array(ids, dtype=np.int64),
            np.array([len(nodes), distinct], dtype=np.int64))


# ---------------------------------------------------------------------------------
# Several jumps (modeling_flashmap.py, draft / embed_state / mix_state;
# flashmap/vllm/model.py, _embed_state and the jump loop)
# ---------------------------------------------------------------------------------


def softmax(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def state_posterior(state: np.ndarray, s: float) -> np.ndarray:
    """The posterior over tokens of a state at time s (modeling_flashmap.py, embed_state):
    softmax(state * s / max(1 - s, 1e-3)^2), rows over the vocabulary."""
    return softmax(np.asarray(state, dtype=np.float64) * (s / max(1.0 - s, 1e-3) ** 2))


def jump_state(state: np.ndarray, delta: np.ndarray, s: float, t: float) -> np.ndarray:
    """The state moved from s to t toward the DiT's distribution delta
    (modeling_flashmap.py, draft): ((1 - t) state + (t - s) delta) / (1 - s)."""
    return ((1.0 - t) * np.asarray(state, dtype=np.float64) + (t - s) * np.asarray(delta, dtype=np.float64)) / (1.0 - s)


def embed_state(cfg: Config, W: dict, C: Constants, E, state: np.ndarray, s: float, t: float) -> np.ndarray:
    """The DiT input of a vocabulary-sized state (rows, V) jumping from s to t, before
    x_embed: state_norm(posterior @ E) + gate * noise_norm(state @ E), the posterior
    softmax(state * s / max(1 - s, 1e-3)^2) (uniform at s = 0, whose embedding is the
    constant u), gate = noise_gate * (t - s) ("jump") or noise_gate ("constant")."""
    E64 = _f64(E)
    if s == 0:
        post = np.broadcast_to(C.uniform, (state.shape[0], C.uniform.shape[0]))
    else:
        post = rms_norm(state_posterior(state, s) @ E64, W["state_norm.weight"], cfg.rms_norm_eps)
    jump = 1.0 if cfg.noise_gate_constant else t - s
    gate = float(np.asarray(W["noise_gate"], dtype=np.float64).reshape(-1)[0]) * jump
    return post + gate * rms_norm(state @ E64, W["noise_norm.weight"], cfg.rms_norm_eps)


def full_logits_of(C: Constants, W: dict, LM, hidden: np.ndarray) -> np.ndarray:
    """The target LM head over the DiT head: LM @ (W_head h + b_head), every token --
    what the full-vocabulary folded head computes (the fold identity)."""
    return (hidden @ _f64(W["head.weight"]).T + _f64(W["head.bias"])) @ _f64(LM).T


def draft_requests_multi(cfg: Config, W: dict, C: Constants, E, LM, ctx_kv: list, anchor_pos: list,
                         seeds: list, num_steps: int, noise_scale: float = 1.0) -> np.ndarray:
    """modeling_flashmap.py, FlashMapDraftModel.draft with num_steps jumps on the printed
    grid (configuration_flashmap.py, DEFAULT_JUMP_GRIDS): the state starts as V-wide
    noise keyed like the one-jump noise (reading R8); each jump s -> t embeds the state
    (embed_state), runs the DiT with the modulations of (s, t), and, before t = 1,
    moves the state to ((1 - t) state + (t - s) softmax(full logits)) / (1 - s).
    Returns the last jump's final AdaLN output (n_req, K, D)."""
    K = cfg.block_size
    nreq = len(anchor_pos)
    grid = DEFAULT_JUMP_GRIDS[str(num_steps)]
    positions = np.concatenate([p + 1 + np.arange(K) for p in anchor_pos])
    state = noise_scale * np.concatenate([draft_normals(sd, p + 1 + np.arange(K), cfg.vocab_size)
                                          for sd, p in zip(seeds, anchor_pos)])
    hidden = None
    for s, t in zip(grid[:-1], grid[1:]):
        mods, final, _ = jump_conditioning(cfg, W, s, t)
        x = embed_state(cfg, W, C, E, state, s, t) @ _f64(W["x_embed.weight"]).T + _f64(W["x_embed.bias"])
        for l in range(cfg.num_layers):
            x = dit_layer(cfg, W, l, mods[l], x, positions, [(kc[l], vc[l]) for kc, vc in ctx_kv])
        hidden = layer_norm(x, cfg.layer_norm_eps) * final[0] + final[1]
        if t < 1.0:
            state = jump_state(state, softmax(full_logits_of(C, W, LM, hidden)), s, t)
    return hidden.reshape(nreq, K, -1)
