"""Which keys are attended, checked exactly, on every masked or indexed path:
the causal prefill, the packed variable-length prefill, the pi-Attention key
set and the paged cache (the contiguous decode has its own such tests in
test_decode_gpu.py).

The method: attended keys have K = 0, so every score is 0 and every weight
exactly 1 (2^0 in the kernels), the sums are exact integers in fp32 and
lse = ln(count) to a few ulp; a key too many or too few moves lse by about
1/count, and the checks separate count from count +- 1.  V[:, 0] = 1 on every
attended key and V[:, 1] = 1 only on probe keys (the edges of tiles, chunks,
pages and the other places where a kernel switches how it addresses keys), so
out[1] = #probes attended / count exactly: a probe dropped or read twice
moves it by 1/count.  Keys that must not be attended are NaN wherever a test
can make them so (past a sequence's end, outside the pi-Attention set,
unreferenced pool rows): reading one turns the row into NaN.

Definitions: the Attention glossary (jisaku.com/glossary/attention, "basic
concepts and operating principle") for the attended set as the keys a
query's softmax runs over; the pi-Attention explainer (gist.science,
technical summary section 2A) for its window plus periodic skips.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_decode_04_b300 import synth, ta

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAN = float("nan")


def _assert_counts(lse, counts, what):
    lse = np.asarray(lse, dtype=np.float64)
    counts = np.asarray(counts, dtype=np.float64)
    assert np.all(np.isfinite(lse)), f"{what}: non-finite lse (a masked key was read)"
    err = np.abs(lse - np.log(counts))
    # neighbours ln(n +- 1) are at least 1/(n+1) away; 1e-5 separates them up to n = 5e4
    assert counts.max() < 5e4
    bad = err >= 1e-5
    assert not bad.any(), f"{what}: {int(bad.sum())} rows off, first count {counts[bad][0]}, err {err[bad][0]:.3g}"


def _assert_probes(out, frac, counts, what):
    out = np.asarray(out, dtype=np.float64)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output (a masked key was read)"
    assert np.all(np.abs(out[..., 0] - 1.0) < 1e-6), f"{what}: weights do not sum to one"
    err = np.abs(out[..., 1] - frac)
    bad = err >= 0.25 / np.asarray(counts, dtype=np.float64)
    assert not bad.any(), f"{what}: probe fraction off in {int(bad.sum())} rows"
    assert np.all(out[..., 2:] == 0.0), f"{what}: a value column that is zero everywhere is not"


# ------------------------------------------------------------ causal prefill

def _prefill_probe_keys(S):
    """Key 0, the last key, the first and last key of every 128-key tile and a
    few keys inside tiles."""
    p = {0, S - 1}
    for t in range(0, S, 128):
        p.update({t, min(S - 1, t + 127)})
    p.update(range(5, S, 997))
    return np.array(sorted(p))


def _prefill_fractions(probes, S):
    """out_i[1] = #{probes <= i} / (i + 1) for every row i."""
    marks = np.zeros(S)
    marks[probes] = 1.0
    return np.cumsum(marks) / np.arange(1, S + 1)


def test_prefill_causal_attends_keys_0_to_i_exactly_s16384():
    """Every row of S = 16384: row i attends exactly keys 0..i (lse = ln(i+1),
    6.1e-5 between neighbours at the last row), probes on every tile edge."""
    B, H, Hkv, S, D = 1, 4, 2, 16384, 128
    g = torch.Generator().manual_seed(11)
    q = torch.randn(B, H, S, D, generator=g).to(torch.bfloat16)
    k = torch.zeros(B, Hkv, S, D, dtype=torch.bfloat16)
    v = torch.zeros(B, Hkv, S, D, dtype=torch.bfloat16)
    v[..., 0] = 1.0
    probes = _prefill_probe_keys(S)
    v[:, :, probes, 1] = 1.0
    out, lse = ta.prefill_causal(q.to(DEV), k.to(DEV), v.to(DEV), scale=0.088, out_dtype=torch.float32)
    torch.cuda.synchronize()
    counts = np.arange(1, S + 1)
    for h in range(H):
        _assert_counts(lse[0, h].cpu().numpy(), counts, f"prefill head {h}")
        _assert_probes(out[0, h].cpu().numpy(), _prefill_fractions(probes, S), counts, f"prefill head {h}")
    assert ta.decode_status() == 0


@pytest.mark.parametrize("S", [1, 127, 128, 129, 255, 256, 257, 383, 385, 1000])
def test_prefill_causal_small_lengths_exact(S):
    """Lengths on both sides of the 128-row tiles and the 256-row CTA pairs, batched
    (two sequences: keys of the next sequence lie past S in memory)."""
    B, H, Hkv, D = 2, 2, 1, 128
    g = torch.Generator().manual_seed(12 + S)
    q = torch.randn(B, H, S, D, generator=g).to(torch.bfloat16)
    k = torch.zeros(B, Hkv, S, D, dtype=torch.bfloat16)
    v = torch.zeros(B, Hkv, S, D, dtype=torch.bfloat16)
    v[..., 0] = 1.0
    probes = _prefill_probe_keys(S)
    v[:, :, probes, 1] = 1.0
    out, lse = ta.prefill_causal(q.to(DEV), k.to(DEV), v.to(DEV), scale=0.3, out_dtype=torch.float32)
    torch.cuda.synchronize()
    counts = np.arange(1, S + 1)
    for b in range(B):
        for h in range(H):
            _assert_counts(lse[b, h].cpu().numpy(), counts, f"S={S} b={b} h={h}")
            _assert_probes(out[b, h].cpu().numpy(), _prefill_fractions(probes, S), counts, f"S={S} b={b} h={h}")


def test_prefill_varlen_attends_only_its_own_sequence_exactly():
    """Packed sequences with lengths around the 128-row tiles: row i of a sequence
    attends exactly its own keys 0..i.  The neighbours' keys also score 0, so a key
    read across a sequence boundary changes the count."""
    lens = [127, 128, 129, 1, 255, 256, 257, 700, 3, 1000]
    H, Hkv, D = 4, 2, 128
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    g = torch.Generator().manual_seed(13)
    q = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    k = torch.zeros(T, Hkv, D, dtype=torch.bfloat16)
    v = torch.zeros(T, Hkv, D, dtype=torch.bfloat16)
    v[..., 0] = 1.0
    counts = np.zeros(T)
    frac = np.zeros(T)
    for s, L in enumerate(lens):
        a = int(cu[s])
        probes = _prefill_probe_keys(L)
        v[a + probes, :, 1] = 1.0
        counts[a:a + L] = np.arange(1, L + 1)
        frac[a:a + L] = _prefill_fractions(probes, L)
    out, lse = ta.prefill_causal_varlen(q.to(DEV), k.to(DEV), v.to(DEV),
                                        torch.tensor(cu, dtype=torch.int32, device=DEV), max(lens), scale=0.2,
                                        out_dtype=torch.float32)
    torch.cuda.synchronize()
    for h in range(H):
        _assert_counts(lse[h].cpu().numpy(), counts, f"packed head {h}")
        _assert_probes(out[:, h].cpu().numpy(), frac, counts, f"packed head {h}")
    assert ta.decode_status() == 0


# ------------------------------------------------------------ pi-Attention key set

def _pi_case(B, Hq, Hkv, S, window, period, lens, probe_every=8):
    """K = 0 on each sequence's attended keys and NaN on every other key; V[:, 0] = 1
    there and V[:, 1] = 1 on probes: list positions 0 and 7 mod 8 (every 8-row group
    edge, so every tile and chunk edge), the last periodic key and the first window
    key (the seam), the first and last keys."""
    D = 128
    k = torch.full((B, Hkv, S, D), NAN, dtype=torch.bfloat16)
    v = torch.full((B, Hkv, S, D), NAN, dtype=torch.bfloat16)
    counts, fracs = [], []
    for b, L in enumerate(lens):
        keys = np.asarray(oracle.pi_key_set(L, window, period), dtype=np.int64)
        i = L - 1
        w0 = max(0, i - window)
        n_skip = int(np.sum(keys < w0))
        pos = np.arange(len(keys))
        probe = (pos % probe_every == 0) | (pos % probe_every == probe_every - 1) | (pos == len(keys) - 1)
        if n_skip > 0:
            probe |= (pos == n_skip - 1) | (pos == n_skip)
        k[b, :, keys] = 0.0
        v[b, :, keys] = 0.0
        v[b, :, keys, 0] = 1.0
        v[b, :, keys[probe], 1] = 1.0
        counts.append(len(keys))
        fracs.append(probe.sum() / len(keys))
    g = torch.Generator().manual_seed(14)
    q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16)
    return q, k, v, np.array(counts), np.array(fracs)


@pytest.mark.parametrize("window,period,S,lens,heads", [
    (4096, 64, 131072, [131072], (32, 8)),          # the benchmark's pi-Attention figure
    (4000, 3, 5003, [5003, 4100], (32, 8)),
    (127, 7, 5003, [5003, 129], (32, 8)),
    (0, 2, 3001, [3001, 2], (32, 8)),
    (500, 120, 9000, [9000, 8999], (32, 8)),
    (16, 64, 20000, [20000, 17], (32, 8)),
    (4000, 3, 5003, [5003, 4100], (2, 2)),          # one query head per KV head: the CUDA-core kernel
    (300, 17, 9000, [9000, 600], (2, 2)),
])
def test_pi_attention_attends_exactly_its_key_set(window, period, S, lens, heads):
    B, (Hq, Hkv) = len(lens), heads
    q, k, v, counts, fracs = _pi_case(B, Hq, Hkv, S, window, period, lens)
    for split in (0, 7):
        out, lse = ta.decode_pi(q.to(DEV), k.to(DEV), v.to(DEV), window, period,
                                seqlens=torch.tensor(lens, dtype=torch.int32, device=DEV), scale=0.1,
                                out_dtype=torch.float32, n_split=split)
        torch.cuda.synchronize()
        for b in range(B):
            _assert_counts(lse[b].cpu().numpy(), np.full(Hq, counts[b]), f"pi b={b} split={split}")
            _assert_probes(out[b].cpu().numpy(), np.full(Hq, fracs[b]), np.full(Hq, counts[b]),
                           f"pi b={b} split={split}")
    assert ta.decode_status() == 0


# ------------------------------------------------------------ paged cache

def _paged_case(lens, page, Hq, Hkv, seed):
    """Contiguous K = 0 / probe V for each sequence's keys, NaN past each length,
    then scattered into a shuffled pool whose unreferenced rows are NaN.  Probes:
    the first and last row of every page and list positions 0 and 7 mod 8."""
    B, D = len(lens), 128
    pages_per_seq = -(-max(lens) // page)
    S = pages_per_seq * page
    k = torch.full((B, Hkv, S, D), NAN, dtype=torch.bfloat16)
    v = torch.full((B, Hkv, S, D), NAN, dtype=torch.bfloat16)
    fracs = []
    for b, L in enumerate(lens):
        j = np.arange(L)
        probe = (j % page == 0) | (j % page == page - 1) | (j % 8 == 0) | (j % 8 == 7) | (j == L - 1)
        k[b, :, :L] = 0.0
        v[b, :, :L] = 0.0
        v[b, :, :L, 0] = 1.0
        v[b, :, j[probe], 1] = 1.0
        fracs.append(probe.sum() / L)
    kp, vp, bt = synth.to_pages(k, v, lens, page, seed=seed, pad_value=NAN)
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16)
    return q, kp, vp, bt, np.array(fracs)


@pytest.mark.parametrize("heads", [(8, 2), (2, 2)], ids=["G4", "G1"])
@pytest.mark.parametrize("page", [8, 16, 64, 128, 120, 1000])
def test_paged_attends_exactly_the_listed_rows(page, heads):
    lens = [1, page - 1 if page > 1 else 1, page, page + 1, 3 * page + 5, 2000, 4097]
    Hq, Hkv = heads
    q, kp, vp, bt, fracs = _paged_case(lens, page, Hq, Hkv, seed=20 + page)
    for split in (0, 9):
        out, lse = ta.decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), bt.to(DEV),
                                   torch.tensor(lens, dtype=torch.int32, device=DEV), scale=0.1,
                                   out_dtype=torch.float32, n_split=split)
        torch.cuda.synchronize()
        for b, L in enumerate(lens):
            _assert_counts(lse[b].cpu().numpy(), np.full(Hq, L), f"paged page={page} b={b}")
            _assert_probes(out[b].cpu().numpy(), np.full(Hq, fracs[b]), np.full(Hq, L), f"paged page={page} b={b}")
    assert ta.decode_status() == 0


def test_paged_full_varlen_b16_64_key_pages_exact():
    """The 16-sequence workload's lengths (1K-32K) in 64-key pages, 32/8 heads."""
    w = synth.WORKLOADS["varlen_b16_32x8_d128_s1k_32k"]
    lens = [int(x) for x in synth.seqlens_for(w)]
    q, kp, vp, bt, fracs = _paged_case(lens, 64, w.Hq, w.Hkv, seed=31)
    out, lse = ta.decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), bt.to(DEV),
                               torch.tensor(lens, dtype=torch.int32, device=DEV), scale=0.1,
                               out_dtype=torch.float32)
    torch.cuda.synchronize()
    for b, L in enumerate(lens):
        # counts above 5e4 cannot occur here (lengths <= 32768)
        _assert_counts(lse[b].cpu().numpy(), np.full(w.Hq, L), f"paged b={b}")
        _assert_probes(out[b].cpu().numpy(), np.full(w.Hq, fracs[b]), np.full(w.Hq, L), f"paged b={b}")
