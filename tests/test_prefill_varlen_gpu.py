"""Causal prefill of packed variable-length sequences on the GPU through the C
ABI: against the float64 oracle, and bit for bit against the batched prefill
when every sequence has the same length (same kernel, other addressing)."""
import numpy as np
import pytest
import torch

import oracle
from long_context_decode_04_b300 import synth, ta
from tests.parity import check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _packed(lens, H, Hkv, seed):
    T = int(sum(lens))
    w = synth.Workload("packed", 5, "prefill", 1, H, Hkv, T, 128, "bf16")
    x = synth.make_inputs(w, seed=seed)
    # [1, H, T, D] -> packed [T, H, D]
    q = x["q"][0].transpose(0, 1).contiguous()
    k = x["k"][0].transpose(0, 1).contiguous()
    v = x["v"][0].transpose(0, 1).contiguous()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    return q, k, v, cu, x["scale"]


def _run(q, k, v, cu, max_len, scale, out_dtype=torch.bfloat16):
    out, lse = ta.prefill_causal_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), max_len, scale=scale,
                                        out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("lens", [[1, 127, 128, 129, 255, 256, 257, 700], [1000, 0, 3, 513], [384] * 3])
def test_varlen_prefill_matches_oracle(lens, out_dtype):
    q, k, v, cu, scale = _packed(lens, 8, 2, seed=1100 + len(lens))
    out, lse = _run(q, k, v, cu, max(lens), scale, out_dtype)
    ro, rl = oracle.prefill_causal_varlen(q, k, v, cu.numpy(), scale)
    check_out(out.float().cpu().numpy().reshape(-1, 128), ro.reshape(-1, 128), bf16=out_dtype == torch.bfloat16)
    check_lse(lse.cpu().numpy(), rl)
    assert ta.decode_status() == 0


def test_equal_lengths_match_the_batched_prefill_bit_for_bit():
    B, S, H, Hkv = 3, 640, 8, 2
    q, k, v, cu, scale = _packed([S] * B, H, Hkv, seed=1200)
    out, lse = _run(q, k, v, cu, S, scale)
    # the same tokens as [B, H, S, D]
    qb = q.view(B, S, H, 128).permute(0, 2, 1, 3).contiguous().to(DEV)
    kb = k.view(B, S, Hkv, 128).permute(0, 2, 1, 3).contiguous().to(DEV)
    vb = v.view(B, S, Hkv, 128).permute(0, 2, 1, 3).contiguous().to(DEV)
    ob, lb = ta.prefill_causal(qb, kb, vb, scale=scale)
    torch.cuda.synchronize()
    assert torch.equal(out.view(B, S, H, 128).permute(0, 2, 1, 3), ob)
    assert torch.equal(lse.view(H, B, S).permute(1, 0, 2), lb)


def test_offsets_past_max_seqlen_are_flagged_not_followed():
    lens = [300, 900]
    q, k, v, cu, scale = _packed(lens, 4, 1, seed=1300)
    out = torch.full((q.shape[0], 4, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((4, q.shape[0]), 7.0, dtype=torch.float32, device=DEV)
    ta.prefill_causal_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), 512, scale=scale, out=out, lse=lse)
    assert ta.decode_status() & ta.TA_DEVERR_SEQLEN
    # rows past max_seqlen were not written; the rest is correct
    ro, rl = oracle.prefill_causal_varlen(q, k, v, cu.numpy(), scale)
    o = out.float().cpu().numpy()
    check_out(o[:300 + 512].reshape(-1, 128), ro[:300 + 512].reshape(-1, 128), bf16=True)
    assert np.all(o[300 + 512:] == 7.0)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_varlen_32_heads_mixed_lengths(out_dtype):
    rng = np.random.Generator(np.random.PCG64(1400))
    lens = [int(x) for x in rng.integers(1, 4096, size=4, endpoint=True)]
    q, k, v, cu, scale = _packed(lens, 32, 8, seed=1400)
    out, lse = _run(q, k, v, cu, max(lens), scale, out_dtype)
    ro, rl = oracle.prefill_causal_varlen(q, k, v, cu.numpy(), scale)
    check_out(out.float().cpu().numpy().reshape(-1, 128), ro.reshape(-1, 128), bf16=out_dtype == torch.bfloat16)
    check_lse(lse.cpu().numpy(), rl)
