"""The C ABI on the host: the library builds and loads without a GPU, exports every
function include/flashmap.h declares, and rejects bad configurations before touching
a device."""

import os

import pytest

from speculative_decoding_block_context_gb300 import _lib as F
from speculative_decoding_block_context_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_block_context_gb300 import build

    build.build()
    return F.lib()


def test_exports_every_header_function(lib):
    names = F.header_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def test_validate_configs_of_every_workload(lib):
    for wl in syn.WORKLOADS:
        cfg = syn.model_config(wl)
        st = F.flashmap_validate_config(cfg)
        assert st == 0, (wl, F.flashmap_last_error())


@pytest.mark.parametrize(
    "change,status",
    [
        (dict(num_steps=5), 2),  # no printed jump grid for 5 jumps
        (dict(noise_path=2), 1),  # 0 (z L^T) or 1 (folded eigenbasis)
        (dict(noise_path=1, num_steps=2), 2),  # the folded path is a one-jump path
        (dict(num_steps=2, vocab_size=1020), 2),  # the state GEMM wants V % 8 == 0
        (dict(num_steps=2, vocab_size=400000, draft_vocab_size=512), 2),  # a state row spans <= 8 CTAs
        (dict(hidden=100), 1),  # hidden != heads * head_dim
        (dict(head_dim=48, hidden=4 * 48), 2),
        (dict(page_size=8), 2),
        (dict(block_size=32), 2),
        (dict(vocab_size=0), 1),
        (dict(act_dtype="f32", weight_dtype="bf16"), 1),
        (dict(act_dtype="f32", weight_dtype="e4m3"), 1),  # e4m3 weights need bf16 activations
        (dict(act_dtype="bf16", weight_dtype="e4m3", kv_dtype="bf16", intermediate=392), 2),  # not a multiple of 16
        (dict(act_dtype="f32", weight_dtype="f32", kv_dtype="e4m3"), 1),  # an e4m3 pool needs bf16 activations
        (dict(act_dtype="bf16", weight_dtype="bf16", kv_dtype="f32"), 1),
        (dict(time_embed_dim=63), 1),
        (dict(rope_theta=-1.0), 1),
    ],
)
def test_invalid_configs_are_rejected_with_a_message(lib, change, status):
    cfg = syn.model_config("tiny_fp32")
    cfg.update(change)
    assert F.flashmap_validate_config(cfg) == status
    assert F.flashmap_last_error()


def test_pool_bytes_layout(lib):
    cfg = syn.model_config("small_bf16")
    n = F.flashmap_pool_bytes(cfg, 10)
    assert n == cfg["num_layers"] * 2 * 10 * cfg["num_heads"] * cfg["page_size"] * cfg["head_dim"] * 2
    with pytest.raises(F.FlashmapError):
        F.flashmap_pool_bytes(cfg, 0)


def test_pool_bytes_per_context_row_matches_the_pages(lib):
    """48 KB per committed row for a 6-layer, 2048-wide bf16 map (the pages' figure)."""
    with open(os.path.join(GOLDEN, "context_row_bytes.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for L, D, el, want in (map(int, r) for r in rows):
        cfg = syn.model_config("qwen3_8b_bs1")
        cfg.update(num_layers=L, hidden=D, num_heads=D // 128, head_dim=128,
                   act_dtype="bf16" if el == 2 else "f32", weight_dtype="bf16" if el == 2 else "f32")
        P = cfg["page_size"]
        assert F.flashmap_pool_bytes(cfg, 1) // P == want


def test_null_model_calls_fail_cleanly(lib):
    import ctypes

    n = ctypes.c_size_t()
    assert lib.flashmap_workspace_size(None, 1, 1, ctypes.byref(n)) == 1
    assert lib.flashmap_free(None) == 0
    assert lib.flashmap_draft_block(None, None, 1, None, None, None, None, 1, None, 1.0, None, None, None, 0,
                                    None) == 1


def test_new_entry_points_reject_null_arguments_before_any_device_work(lib):
    """The draft with a deferred write, the GEMM chain hook, the wait-timeout probe and
    the static sampler refuse NULL arguments with E_INVALID and a message (no model, no
    device needed)."""
    import ctypes

    b, n = ctypes.c_int64(), ctypes.c_int32()
    assert lib.flashmap_draft_block_with_write(None, None, None, 1, None, None, None, None, 1, None, 1.0, None,
                                               None, None, 0, None) == 1
    assert F.flashmap_last_error()
    assert lib.flashmap_profile_gemm_chain(None, 1, 17, None, None, 0, ctypes.byref(b), ctypes.byref(n), None) == 1
    assert lib.flashmap_debug_wait_timeout(None, 1000000, None) == 1
    assert lib.flashmap_sample_logits_static(None, 1, None, None, None, None, None, 0, None, None) == 1


def test_e4m3_pool_is_half_the_bf16_pool(lib):
    cfg = syn.model_config("qwen3_8b_bs32_kv8")
    assert cfg["kv_dtype"] == "e4m3"
    n8 = F.flashmap_pool_bytes(cfg, 7)
    assert n8 * 2 == F.flashmap_pool_bytes(dict(cfg, kv_dtype="bf16"), 7)
    L, nh, P, hd = (cfg[k] for k in ("num_layers", "num_heads", "page_size", "head_dim"))
    assert n8 == L * 2 * 7 * nh * P * hd
