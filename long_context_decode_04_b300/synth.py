"""Seeded synthetic inputs for the attention workloads.

This module holds the workload shapes and the random-number recipe, and
nothing of the attention arithmetic: both the CUDA path (through the tests
and the benchmark) and the float64 oracle draw their inputs from here, so
they see bit-identical tensors.

Recipe
------
* Values are i.i.d. N(0, 1) drawn with numpy's PCG64 generator.  A tensor
  is cut into blocks of ``BLOCK`` elements; block ``i`` of tensor ``name``
  uses ``SeedSequence([seed, tag(name), i])``, so the values do not depend
  on how many threads draw them.
* Draws are float32 and are rounded to bfloat16 round-to-nearest-even when
  the workload is bf16 (torch's ``.to(torch.bfloat16)``).
* The seed of a workload is ``1000 + its index`` in ``WORKLOADS`` (1-based).

The shapes are those of a Llama-3.1-8B attention layer (32 query heads,
8 KV heads, head dim 128), the model the Tree Attention explainer
(aibr.jp/archives/143699, section 4) evaluates decode on.  No weights or
datasets are involved: only the shapes are borrowed.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

BLOCK = 1 << 24  # elements per independently seeded block

_TAGS = {"q": 1, "k": 2, "v": 3, "seqlens": 4, "peak_rows": 5, "pages": 6}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention workload, named by what it is."""

    name: str
    index: int          # 1-based position; the seed is 1000 + index
    kind: str           # "decode" or "prefill"
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    dtype: str          # "f32" or "bf16" (q, K, V and the output)
    varlen: tuple | None = None   # (lo, hi) inclusive range of per-sequence lengths
    peak_frac: float = 0.0        # fraction of key rows scaled by peak_scale
    peak_scale: float = 1.0
    chunk: int | None = None      # forced split-KV chunk (keys per split)

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


WORKLOADS = {
    w.name: w
    for w in [
        Workload("single_head_d64_s4096_f32", 1, "decode", 1, 1, 1, 4096, 64, "f32"),
        Workload("gqa_32x8_d128_s131072", 2, "decode", 1, 32, 8, 131072, 128, "bf16"),
        Workload("varlen_b16_32x8_d128_s1k_32k", 3, "decode", 16, 32, 8, 32768, 128, "bf16",
                 varlen=(1024, 32768), peak_frac=0.01, peak_scale=8.0),
        Workload("gqa_32x8_d128_s1048576_c256", 4, "decode", 1, 32, 8, 1 << 20, 128, "bf16",
                 chunk=256),
        Workload("causal_prefill_32x8_d128_s16384", 5, "prefill", 1, 32, 8, 16384, 128, "bf16"),
    ]
}


def _normal_f32(seed: int, tag: int, n: int, threads: int | None = None) -> np.ndarray:
    """n float32 N(0,1) draws, block-seeded so the result is thread-count independent."""
    out = np.empty(n, dtype=np.float32)
    nblocks = (n + BLOCK - 1) // BLOCK

    def fill(i: int) -> None:
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, i])))
        lo = i * BLOCK
        hi = min(n, lo + BLOCK)
        out[lo:hi] = rng.standard_normal(hi - lo, dtype=np.float32)

    threads = threads or min(32, os.cpu_count() or 1)
    if nblocks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(nblocks)))
    return out


def normal(shape, dtype: str, seed: int, name: str) -> torch.Tensor:
    """A CPU tensor of i.i.d. N(0,1) values, bf16-rounded when dtype == 'bf16'."""
    n = int(np.prod(shape)) if len(shape) else 1
    a = torch.from_numpy(_normal_f32(seed, _TAGS[name], n)).reshape(shape)
    if dtype == "bf16":
        return a.to(torch.bfloat16)
    if dtype == "f32":
        return a
    raise ValueError(f"unknown dtype {dtype!r}")


def seqlens_for(w: Workload) -> torch.Tensor | None:
    """Per-sequence lengths, uniform on the inclusive range, or None (all S)."""
    if w.varlen is None:
        return None
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, _TAGS["seqlens"]])))
    lo, hi = w.varlen
    return torch.from_numpy(rng.integers(lo, hi, size=w.B, endpoint=True).astype(np.int32))


def peak_row_mask(w: Workload) -> torch.Tensor | None:
    """Boolean [B, Hkv, S]: key rows that are scaled by ``peak_scale``."""
    if w.peak_frac <= 0:
        return None
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, _TAGS["peak_rows"]])))
    return torch.from_numpy(rng.random((w.B, w.Hkv, w.S)) < w.peak_frac)


def make_inputs(w: Workload, *, seed: int | None = None, S: int | None = None,
                B: int | None = None, pad_value: float | None = None) -> dict:
    """CPU tensors for workload ``w`` (optionally with a smaller S or B).

    Returns dict(q, k, v, seqlens, scale).  Decode layout: q [B,Hq,D],
    K/V [B,Hkv,S,D].  Prefill layout: q [B,Hq,S,D], K/V [B,Hkv,S,D].
    ``pad_value`` (e.g. NaN) overwrites K/V rows at or beyond each
    sequence's length, so that a kernel touching a masked key shows it.
    """
    seed = w.seed if seed is None else seed
    S = w.S if S is None else S
    B = w.B if B is None else B
    shape_q = (B, w.Hq, w.D) if w.kind == "decode" else (B, w.Hq, S, w.D)
    q = normal(shape_q, w.dtype, seed, "q")
    k = normal((B, w.Hkv, S, w.D), w.dtype, seed, "k")
    v = normal((B, w.Hkv, S, w.D), w.dtype, seed, "v")
    seqlens = None
    if w.varlen is not None:
        wl = dataclasses.replace(w, B=B, S=S)
        seqlens = seqlens_for(wl)
        if S < w.S:
            # keep the length distribution's shape when a test shrinks S
            seqlens = torch.clamp((seqlens.long() * S) // w.S, min=1).to(torch.int32)
    if w.peak_frac > 0:
        mask = peak_row_mask(dataclasses.replace(w, B=B, S=S))
        k[mask] = (k[mask].float() * w.peak_scale).to(k.dtype)
    if pad_value is not None and seqlens is not None:
        for b in range(B):
            k[b, :, int(seqlens[b]):, :] = pad_value
            v[b, :, int(seqlens[b]):, :] = pad_value
    return {"q": q, "k": k, "v": v, "seqlens": seqlens, "scale": w.scale}


def to_pages(k: torch.Tensor, v: torch.Tensor, seqlens, page_size: int, *, seed: int = 7,
             extra_pages: int = 3, pad_value: float | None = None):
    """Scatter contiguous K/V [B, Hkv, S, D] into a shuffled page pool.

    Returns (k_pages, v_pages [num_pages, Hkv, page_size, D], block_table
    [B, pages_per_seq] int32).  Sequence b's key j goes to row j % page_size
    of page block_table[b, j // page_size]; physical pages are a seeded
    permutation, ``extra_pages`` pages belong to no sequence, and block-table
    slots past a sequence's last page point at one of them.  ``pad_value``
    (e.g. NaN) fills every pool row that holds no attended key, so a kernel
    reading one shows it.  Pure data movement: no attention arithmetic.
    """
    B, Hkv, S, D = k.shape
    lens = [S] * B if seqlens is None else [int(x) for x in seqlens]
    pages_per_seq = (S + page_size - 1) // page_size
    used = [(L + page_size - 1) // page_size for L in lens]
    num_pages = sum(used) + extra_pages
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _TAGS["pages"], page_size])))
    perm = rng.permutation(num_pages)
    fill = 0.0 if pad_value is None else pad_value
    kp = torch.full((num_pages, Hkv, page_size, D), fill, dtype=k.dtype)
    vp = torch.full((num_pages, Hkv, page_size, D), fill, dtype=v.dtype)
    spare = [int(x) for x in perm[sum(used):]] or [int(perm[0])]
    table = torch.empty((B, pages_per_seq), dtype=torch.int32)
    nxt = 0
    for b in range(B):
        for pg in range(pages_per_seq):
            if pg < used[b]:
                phys = int(perm[nxt])
                nxt += 1
                j0 = pg * page_size
                n = min(page_size, lens[b] - j0)
                kp[phys, :, :n] = k[b, :, j0:j0 + n]
                vp[phys, :, :n] = v[b, :, j0:j0 + n]
            else:
                phys = spare[pg % len(spare)]
            table[b, pg] = phys
    return kp, vp, table


def to_e4m3(x: torch.Tensor):
    """Quantise K or V [B, Hkv, S, D] to FP8 E4M3 with one scale per (sequence,
    KV head): scale = max|x| / 448 (the largest finite E4M3), bits = RNE of
    x / scale (torch's float8_e4m3fn cast).  Returns (uint8 bit patterns,
    float32 scales [B*Hkv]).  Input generation only."""
    B, Hkv = x.shape[:2]
    xf = x.float()
    amax = xf.abs().amax(dim=(2, 3)).clamp_min(1e-30)
    sc = (amax / 448.0).to(torch.float32)
    bits = (xf / sc.view(B, Hkv, 1, 1)).to(torch.float8_e4m3fn).view(torch.uint8)
    return bits.contiguous(), sc.reshape(-1).contiguous()


_E2M1_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_codes(y: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code of each value (ties to the even code, magnitudes above
    6 saturate to 6): sign in bit 3, magnitude index in bits 0-2."""
    a = np.minimum(np.abs(y), 6.0)
    idx = np.searchsorted(_E2M1_MAGS, a)            # first magnitude >= a
    idx = np.clip(idx, 1, 7)
    lo, hi = _E2M1_MAGS[idx - 1], _E2M1_MAGS[idx]
    pick_hi = (a - lo > hi - a) | ((a - lo == hi - a) & (idx % 2 == 0))
    code = np.where(pick_hi, idx, idx - 1)
    code = np.where(a == 0, 0, code)
    return (code | np.where(y < 0, 8, 0)).astype(np.uint8)


def to_nvfp4(x: torch.Tensor):
    """Quantise K or V [B, Hkv, S, D] to NVFP4: one fp32 factor per (sequence,
    KV head) = max|x| / (6 * 448), one E4M3 scale per 16 consecutive elements
    of a row = RNE of (block max|x| / 6) / factor (torch's float8_e4m3fn
    cast), elements = nearest E2M1 of x / (scale * factor).  Returns (codes
    [B, Hkv, S, D/2] uint8 with element 2i in the low nibble, scales [B, Hkv,
    S, D/16] uint8, factors [B*Hkv] float32).  Input generation only."""
    B, Hkv, S, D = x.shape
    xf = x.float()
    amax = xf.abs().amax(dim=(2, 3)).clamp_min(1e-30)
    fac = (amax / (6.0 * 448.0)).to(torch.float32)
    blocks = xf.reshape(B, Hkv, S, D // 16, 16)
    bmax = blocks.abs().amax(dim=-1)
    sc = (bmax / 6.0 / fac.view(B, Hkv, 1, 1)).to(torch.float8_e4m3fn)
    sc_val = sc.float().clamp_min(2.0 ** -9)  # a zero scale only occurs for an all-zero block
    y = (blocks / (sc_val.unsqueeze(-1) * fac.view(B, Hkv, 1, 1, 1))).reshape(B, Hkv, S, D).numpy()
    codes = _e2m1_codes(y)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return (torch.from_numpy(np.ascontiguousarray(packed)), sc.view(torch.uint8).contiguous(),
            fac.reshape(-1).contiguous())
