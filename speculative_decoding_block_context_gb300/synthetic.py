"""Seeded synthetic inputs for the FlashMap block-draft step.

This module only draws numbers: model weights with the shapes of a FlashMap
drafter, the target's embedding and LM head, a draft-vocabulary ranking, and the
per-request inputs of a draft step (context lengths, page tables, anchors, seeds,
temperatures, verify windows). It holds none of the method's arithmetic. Tests and
bench.py feed the same draws to the CUDA library and to the CPU oracle.

Distributions (no public dataset or checkpoint is involved): linear weights
N(0, 1/fan_in); the embedding E N(0, 0.02^2); the LM head N(0, 1/H); norm weights
1 + 0.1 N(0, 1); biases 0.02 N(0, 1); noise_gate 1; the ranking a random
permutation of the vocabulary; target hidden states N(0, 1); anchors uniform over
the vocabulary; request seeds uniform in [0, 2^63). Values are drawn in float32 with
torch generators on the target device and rounded once to the activation dtype,
so every consumer sees the same numbers.
"""

from __future__ import annotations

import math

import torch

# Model shapes. "tiny" is the fp32 check case; "qwen3_8b" is a drafter sized for a
# Qwen3-8B target (target_hidden 4096 read from 3 target layers, DiT 5 x 4096,
# 32 heads x 128, MLP 12288, vocabulary 151936 with a 32768-token draft vocabulary);
# "small" spans several GEMM tiles with ragged tails at a size the oracle finishes
# in seconds.
MODELS = {
    "tiny": dict(target_hidden=256, num_target_layers=3, hidden=128, num_layers=2, num_heads=4,
                 head_dim=32, intermediate=384, cond_dim=64, time_embed_dim=64, block_size=4,
                 vocab_size=1024, draft_vocab_size=512, page_size=16, rope_theta=1e4,
                 act_dtype="f32", weight_dtype="f32", max_position=4096),
    "small": dict(target_hidden=384, num_target_layers=3, hidden=320, num_layers=2, num_heads=5,
                  head_dim=64, intermediate=704, cond_dim=96, time_embed_dim=64, block_size=16,
                  vocab_size=5000, draft_vocab_size=1234, page_size=16, rope_theta=1e6,
                  act_dtype="bf16", weight_dtype="bf16", max_position=4096),
    # one DiT layer at the Qwen3-8B width with a small vocabulary: a case for profiling
    # the cross-attention on ~1 GB of context without the full model's weights
    "probe": dict(target_hidden=1024, num_target_layers=1, hidden=4096, num_layers=1, num_heads=32,
                  head_dim=128, intermediate=1024, cond_dim=64, time_embed_dim=64, block_size=16,
                  vocab_size=2048, draft_vocab_size=0, page_size=16, rope_theta=1e6,
                  act_dtype="bf16", weight_dtype="bf16", max_position=8192),
    "qwen3_8b": dict(target_hidden=4096, num_target_layers=3, hidden=4096, num_layers=5,
                     num_heads=32, head_dim=128, intermediate=12288, cond_dim=256,
                     time_embed_dim=256, block_size=16, vocab_size=151936,
                     draft_vocab_size=32768, page_size=16, rope_theta=1e6,
                     act_dtype="bf16", weight_dtype="bf16", max_position=40960),
}
COMMON = dict(time_scale=1000.0, rms_norm_eps=1e-6, qk_norm_eps=1e-5, layer_norm_eps=1e-6,
              noise_gate_constant=0, num_steps=1)

# Workloads. ctx: committed context length per request before the step.
# window: the step writes a verify window of block_size + 1 columns at positions
# ctx..ctx+block_size with 1..block_size of them committed; the anchor then sits
# at ctx + commit. prefill: the context itself is written by the library from
# synthetic target hidden states; otherwise it is drawn as N(0, 1) keys/values.
WORKLOADS = {
    "tiny_fp32": dict(model="tiny", bs=1, ctx=("fixed", 64), prefill=True, window=False,
                      temps=("greedy",), full_scatter=False, seed=0),
    "small_bf16": dict(model="small", bs=3, ctx=("list", [37, 300, 129]), prefill=True,
                       window=True, temps=("mix", 0.5, 1.2), full_scatter=True, seed=11),
    "attn_probe": dict(model="probe", bs=16, ctx=("fixed", 4096), prefill=False, window=False,
                       temps=("greedy",), full_scatter=False, seed=6),
    "attn_probe_kv8": dict(model="probe", bs=16, ctx=("fixed", 4096), prefill=False, window=False,
                           temps=("greedy",), full_scatter=False, seed=6, kv_dtype="e4m3"),
    "qwen3_8b_bs1": dict(model="qwen3_8b", bs=1, ctx=("fixed", 2048), prefill=True, window=True,
                         temps=("all", 1.0), full_scatter=False, seed=2),
    "qwen3_8b_bs32": dict(model="qwen3_8b", bs=32, ctx=("uniform", 512, 8192), prefill=False,
                          window=False, temps=("mix", 0.5, 1.2), full_scatter=False, seed=3),
    "qwen3_8b_bs128": dict(model="qwen3_8b", bs=128, ctx=("loguniform", 16, 32768),
                           prefill=False, window=True, temps=("mix", 0.5, 1.2),
                           full_scatter=True, seed=4),
    "qwen3_8b_fp8_bs64": dict(model="qwen3_8b", bs=64, ctx=("uniform", 1024, 16384),
                              prefill=False, window=False, temps=("greedy",),
                              full_scatter=False, seed=5, weight_dtype="e4m3"),
    # several jumps on the printed grids (a vocabulary-sized state between jumps)
    "tiny_fp32_2jump": dict(model="tiny", bs=1, ctx=("fixed", 64), prefill=True, window=False,
                            temps=("greedy",), full_scatter=False, seed=20, num_steps=2),
    "small_bf16_3jump": dict(model="small", bs=3, ctx=("list", [37, 300, 129]), prefill=True,
                             window=True, temps=("mix", 0.5, 1.2), full_scatter=False, seed=21,
                             num_steps=3),
    "qwen3_8b_bs1_2jump": dict(model="qwen3_8b", bs=1, ctx=("fixed", 2048), prefill=True, window=True,
                               temps=("all", 1.0), full_scatter=False, seed=2, num_steps=2),
    # the folded-noise eigenbasis (noise_path 1): one GEMM through M instead of z L^T
    "tiny_fp32_folded": dict(model="tiny", bs=1, ctx=("fixed", 64), prefill=True, window=False,
                             temps=("greedy",), full_scatter=False, seed=30, noise_path=1),
    "small_bf16_folded": dict(model="small", bs=3, ctx=("list", [37, 300, 129]), prefill=True,
                              window=True, temps=("mix", 0.5, 1.2), full_scatter=False, seed=31,
                              noise_path=1),
    "qwen3_8b_bs1_folded": dict(model="qwen3_8b", bs=1, ctx=("fixed", 2048), prefill=True, window=True,
                                temps=("all", 1.0), full_scatter=False, seed=2, noise_path=1),
    # tree drafting: 4 candidate blocks per request (greedy), the verify tree of width 16
    "qwen3_8b_bs1_tree4": dict(model="qwen3_8b", bs=1, ctx=("fixed", 2048), prefill=True, window=True,
                               temps=("greedy",), full_scatter=False, seed=2, tree=(4, 16)),
    "qwen3_8b_bs32_tree4": dict(model="qwen3_8b", bs=32, ctx=("uniform", 512, 8192), prefill=False,
                                window=False, temps=("greedy",), full_scatter=False, seed=3, tree=(4, 16)),
    # e4m3 draft KV pool (keys and values stored with scale 1, fp8 queries per head)
    "small_bf16_kv8": dict(model="small", bs=3, ctx=("list", [37, 300, 129]), prefill=True,
                           window=True, temps=("mix", 0.5, 1.2), full_scatter=False, seed=12,
                           kv_dtype="e4m3"),
    "qwen3_8b_bs32_kv8": dict(model="qwen3_8b", bs=32, ctx=("uniform", 512, 8192), prefill=False,
                              window=False, temps=("mix", 0.5, 1.2), full_scatter=False, seed=3,
                              kv_dtype="e4m3"),
    "qwen3_8b_bs128_kv8": dict(model="qwen3_8b", bs=128, ctx=("loguniform", 16, 32768),
                               prefill=False, window=True, temps=("mix", 0.5, 1.2),
                               full_scatter=True, seed=4, kv_dtype="e4m3"),
}

MODEL_SEED = 1234  # one weight draw per model shape, shared by its workloads


def model_config(workload: str) -> dict:
    wl = WORKLOADS[workload]
    cfg = dict(MODELS[wl["model"]])
    cfg.update(COMMON)
    if "weight_dtype" in wl:
        cfg["weight_dtype"] = wl["weight_dtype"]
    cfg["kv_dtype"] = wl.get("kv_dtype", cfg["act_dtype"])
    cfg["num_steps"] = wl.get("num_steps", 1)
    cfg["noise_path"] = wl.get("noise_path", 0)
    return cfg


def torch_dtype(name: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}[name]


def weight_shapes(cfg: dict) -> dict:
    """Canonical weight names (the module names of the reference model) -> shape."""
    H, Lt, D = cfg["target_hidden"], cfg["num_target_layers"], cfg["hidden"]
    C, Te, F, hd = cfg["cond_dim"], cfg["time_embed_dim"], cfg["intermediate"], cfg["head_dim"]
    s = {
        "fc.weight": (D, Lt * H), "hidden_norm.weight": (D,),
        "anchor_proj.weight": (D, H), "anchor_proj.bias": (D,), "anchor_norm.weight": (D,),
        "state_norm.weight": (H,), "noise_norm.weight": (H,), "noise_gate": (1,),
        "x_embed.weight": (D, H), "x_embed.bias": (D,),
        "final_adaln.linear.weight": (3 * D, C), "final_adaln.linear.bias": (3 * D,),
        "head.weight": (H, D), "head.bias": (H,),
    }
    for te in ("time_embed", "jump_embed"):
        s[f"{te}.linear_1.weight"] = (C, Te)
        s[f"{te}.linear_1.bias"] = (C,)
        s[f"{te}.linear_2.weight"] = (C, C)
        s[f"{te}.linear_2.bias"] = (C,)
    for l in range(cfg["num_layers"]):
        p = f"layers.{l}"
        for norm in ("self_attn_adaln", "cross_attn_adaln", "mlp_adaln"):
            s[f"{p}.{norm}.linear.weight"] = (3 * D, C)
            s[f"{p}.{norm}.linear.bias"] = (3 * D,)
        for att in ("self_attn", "cross_attn"):
            for proj in ("q_proj", "k_proj", "v_proj", "o_proj"):
                s[f"{p}.{att}.{proj}.weight"] = (D, D)
            s[f"{p}.{att}.q_norm.weight"] = (hd,)
            s[f"{p}.{att}.k_norm.weight"] = (hd,)
        s[f"{p}.mlp.fc1.weight"] = (F, D)
        s[f"{p}.mlp.fc1.bias"] = (F,)
        s[f"{p}.mlp.fc2.weight"] = (D, F)
        s[f"{p}.mlp.fc2.bias"] = (D,)
    return s


def make_model(cfg: dict, device, seed: int = MODEL_SEED):
    """Weights (name -> tensor in the activation dtype), the target's embedding E and
    LM head (V, H), and the draft-vocabulary ranking (V,) int64, on ``device``."""
    dt = torch_dtype(cfg["act_dtype"])
    g = torch.Generator(device=device).manual_seed(seed)
    W = {}
    for name, shape in weight_shapes(cfg).items():
        if name == "noise_gate":
            W[name] = torch.ones(shape, device=device, dtype=dt)
            continue
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if name.endswith("norm.weight"):
            x = 1.0 + 0.1 * x
        elif name.endswith(".bias"):
            x = 0.02 * x
        else:  # linear weight (out, in): N(0, 1/fan_in)
            x = x * (1.0 / math.sqrt(shape[1]))
        W[name] = x.to(dt)
    V, H = cfg["vocab_size"], cfg["target_hidden"]
    E = (0.02 * torch.randn((V, H), generator=g, device=device)).to(dt)
    LM = (torch.randn((V, H), generator=g, device=device) / math.sqrt(H)).to(dt)
    ranking = torch.randperm(V, generator=g, device=device).to(torch.int64)
    return W, E, LM, ranking


def _draw_lengths(spec, bs: int, g: torch.Generator) -> list:
    kind = spec[0]
    if kind == "fixed":
        return [int(spec[1])] * bs
    if kind == "list":
        return [int(x) for x in spec[1]][:bs]
    if kind == "uniform":
        lo, hi = spec[1], spec[2]
        return [int(x) for x in torch.randint(lo, hi + 1, (bs,), generator=g)]
    if kind == "loguniform":
        lo, hi = math.log(spec[1]), math.log(spec[2])
        u = torch.rand((bs,), generator=g, dtype=torch.float64)
        return [int(math.floor(math.exp(lo + float(x) * (hi - lo)))) for x in u]
    raise ValueError(spec)


def make_requests(workload: str, device, *, bs: int | None = None, seed: int | None = None):
    """Per-request inputs of one draft step for ``workload`` (host-side integer draws
    from a CPU generator; large float tensors on ``device``).

    Returns a dict with python lists (ctx, commit, anchor_pos, ...) and device
    tensors (req_to_page, req_pool_idx, anchor_ids, seeds, temperature, greedy, ...).
    """
    wl = WORKLOADS[workload]
    cfg = model_config(workload)
    bs = wl["bs"] if bs is None else bs
    seed = wl["seed"] if seed is None else seed
    g = torch.Generator().manual_seed(seed)
    K, P, V = cfg["block_size"], cfg["page_size"], cfg["vocab_size"]
    ctx = _draw_lengths(wl["ctx"], bs, g)
    if wl["window"]:
        commit = [int(x) for x in torch.randint(1, K + 1, (bs,), generator=g)]
    else:
        commit = [0] * bs
    anchor_pos = [c + m for c, m in zip(ctx, commit)]
    # Room for the context, the verify window and the next block.
    pages_per_req = [(max(p, c + K + 1) + K + 2 + P - 1) // P for p, c in zip(anchor_pos, ctx)]
    rows = bs + 3  # more page-table rows than requests: req_pool_idx is an indirection
    max_pages = max(pages_per_req)
    num_pages = sum(pages_per_req) + 7
    perm = torch.randperm(num_pages, generator=g)
    req_pool_idx = torch.randperm(rows, generator=g)[:bs].to(torch.int32)
    req_to_page = torch.full((rows, max_pages), -1, dtype=torch.int32)
    off = 0
    for b in range(bs):
        n = pages_per_req[b]
        req_to_page[int(req_pool_idx[b]), :n] = perm[off : off + n].to(torch.int32)
        off += n
    anchor_ids = torch.randint(0, V, (bs,), generator=g, dtype=torch.int64)
    seeds = torch.randint(0, 2**63 - 1, (bs,), generator=g, dtype=torch.int64)
    kind = wl["temps"][0]
    if kind == "greedy":
        temperature = torch.zeros(bs)
        greedy = torch.ones(bs, dtype=torch.uint8)
    elif kind == "all":
        temperature = torch.full((bs,), float(wl["temps"][1]))
        greedy = torch.zeros(bs, dtype=torch.uint8)
    else:
        lo, hi = wl["temps"][1], wl["temps"][2]
        temperature = lo + (hi - lo) * torch.rand((bs,), generator=g)
        greedy = (torch.arange(bs) % 2 == 0).to(torch.uint8)  # half greedy
        temperature = torch.where(greedy.bool(), torch.zeros(bs), temperature)
    out = dict(
        bs=bs, ctx=ctx, commit=commit, anchor_pos=anchor_pos, num_pages=num_pages,
        window=K + 1 if wl["window"] else 0,
        req_to_page=req_to_page.to(device), req_pool_idx=req_pool_idx.to(device),
        anchor_ids=anchor_ids.to(device), seeds=seeds.to(device),
        temperature=temperature.to(torch.float32).to(device), greedy=greedy.to(device),
        step=int(torch.randint(0, 1000, (1,), generator=g)),
        full_scatter=wl["full_scatter"], prefill=wl["prefill"],
        tree=wl.get("tree"),  # (candidates per request, tree width) or None
    )
    dt = torch_dtype(cfg["act_dtype"])
    gd = torch.Generator(device=device).manual_seed(seed + 1000)
    width = cfg["target_hidden"] * cfg["num_target_layers"]
    if wl["prefill"]:
        # Target hidden states of the committed context of each request.
        out["prefill_hidden"] = [
            torch.randn((c, width), generator=gd, device=device).to(dt) for c in ctx
        ]
    if wl["window"]:
        out["window_hidden"] = torch.randn((bs, K + 1, width), generator=gd, device=device).to(dt)
    out["kv_generator_seed"] = seed + 2000
    return out


def fill_pool_random(pool: torch.Tensor, seed: int) -> None:
    """Prefilled context keys/values: N(0, 1) in the pool's dtype, every slot."""
    g = torch.Generator(device=pool.device).manual_seed(seed)
    flat = pool.view(-1)
    chunk = 1 << 28
    for s in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - s)
        if pool.dtype == torch.float8_e4m3fn:  # drawn in float32, stored as e4m3
            flat[s : s + n] = torch.randn((n,), generator=g, device=pool.device).to(pool.dtype)
        else:
            flat[s : s + n] = torch.randn((n,), generator=g, device=pool.device, dtype=pool.dtype)
