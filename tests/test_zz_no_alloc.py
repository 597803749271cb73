"""flashmap_sample_logits_static: sampling without any device allocation.

Some callers cannot allocate device memory (a host runtime that owns all device
memory and hands a plugin only its input and output buffers, for instance). For them
the library keeps the sampler's per-row merge slots in a fixed array of its own. This
checks, through the C ABI, that the entry point draws exactly the tokens that
flashmap_sample_block draws from the same logits, on two calls in a row with
different batch sizes (the array keeps the previous call's contents, which each call
must clear), with rows sampled by one CTA and by several CTAs that merge through the
array, and that batches beyond the array's 8192 rows are refused before anything
runs.
"""

import pytest
import torch

from speculative_decoding_block_context_gb300 import _lib as F
from speculative_decoding_block_context_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _load(draft_vocab):
    from speculative_decoding_block_context_gb300 import build

    build.build()
    cfg = syn.model_config("small_bf16")
    cfg["draft_vocab_size"] = draft_vocab
    W, E, LM, rank = syn.make_model(cfg, "cuda")
    handle = F.flashmap_load_weights(cfg, W, E, LM, rank)
    torch.cuda.synchronize()
    return cfg, handle, E


# Two draft vocabularies: 1234 entries (one CTA per row, scalar loads: 1234 is not a
# multiple of 4) and 4996 (a multiple of 4 above 4096: three CTAs per row on the
# vectorised path, merging through the array's per-row keys and counters).
@pytest.fixture(scope="module", params=[1234, 4996], ids=["vd1234_one_cta_per_row", "vd4996_split_rows"])
def model(request):
    return _load(request.param)


def _inputs(cfg, bs, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    K, D = cfg["block_size"], cfg["hidden"]
    hidden = torch.randn((bs * K, D), generator=g, device="cuda").to(torch.bfloat16)
    anchor_pos = torch.randint(0, 1000, (bs,), generator=g, device="cuda", dtype=torch.int32)
    temperature = 0.5 + torch.rand((bs,), generator=g, device="cuda")
    greedy = (torch.arange(bs, device="cuda") % 3 == 0).to(torch.uint8)
    seeds = torch.randint(0, 2**62, (bs,), generator=g, device="cuda", dtype=torch.int64)
    return hidden, anchor_pos, temperature, greedy, seeds


def test_static_sampler_matches_sample_block_on_two_calls(model):
    """Two calls in a row, the larger batch first: the second call's counters start at
    a lower offset of the array (they follow its bs * K keys), over bytes the first
    call used as keys."""
    cfg, handle, _ = model
    K = cfg["block_size"]
    vd = cfg["draft_vocab_size"]
    ws = torch.empty(F.flashmap_workspace_size(handle, 7, 1), dtype=torch.uint8, device="cuda")
    for call, (bs, step) in enumerate(((7, 7), (3, 8))):
        hidden, anchor_pos, temperature, greedy, seeds = _inputs(cfg, bs, 100 + call)
        want = torch.empty(bs * K, dtype=torch.int64, device="cuda")
        logits = torch.empty((bs * K, vd), dtype=torch.float32, device="cuda")
        F.flashmap_sample_block(handle, bs, hidden, anchor_pos, temperature, greedy, seeds, step, want, logits,
                                None, ws)
        got = torch.full((bs * K,), -1, dtype=torch.int64, device="cuda")
        F.flashmap_sample_logits_static(handle, bs, logits, anchor_pos, temperature, greedy, seeds, step, got)
        torch.cuda.synchronize()
        # same logits, same noise: the same token ids, exactly
        assert torch.equal(got, want), f"call {call}: {got.tolist()} vs {want.tolist()}"
    assert F.flashmap_get_device_error(handle) == 0


def test_static_sampler_refuses_batches_beyond_its_array():
    cfg, handle, _ = _load(1234)
    K = cfg["block_size"]
    bs = 8192 // K + 1
    t = torch.zeros(1, device="cuda")
    with pytest.raises(F.FlashmapError) as err:
        F.flashmap_sample_logits_static(handle, bs, t, t, t, t, t, 0, t)
    assert err.value.status == 1 and "8192" in str(err.value)
