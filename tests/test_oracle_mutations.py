"""Every plausible mistake planted in a copy of the oracle is caught by a pin.

Each case copies oracle/oracle.c to a temporary directory, applies one
textual change (a dropped term, a wrong sign, a wrong index, a swapped
operand), compiles the copy, points the oracle wrapper at it and runs all
pins: at least one must fail.  The shipped oracle is never modified.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = {
    "dropped_scale": ("s[j - j0] = scale * dot;", "s[j - j0] = dot;"),
    "exp_sign_flipped": ("sum += exp(s[j] - m);", "sum += exp(m - s[j]);"),
    "max_not_subtracted_in_lse": ("double lse_v = m + log(sum);", "double lse_v = log(sum);"),
    "log2_instead_of_ln": ("double lse_v = m + log(sum);", "double lse_v = m + log2(sum);"),
    "weights_unnormalised": ("double w = exp(s[j] - lse_v);", "double w = exp(s[j] - m);"),
    "scores_dims_reversed": ("widen(k, kv_dtype, kv_base + (size_t)j * D + d)", "widen(k, kv_dtype, kv_base + (size_t)j * D + (D - 1 - d))"),
    "gqa_index_modulo": ("(size_t)(h / G)) * (size_t)S * D;", "(size_t)(h % job->Hkv)) * (size_t)S * D;"),
    "seqlens_ignored": ("L = job->seqlens ? job->seqlens[b] : S;", "L = S;"),
    "causal_excludes_diagonal": ("L = i + 1;", "L = i;"),
    "causal_one_too_many": ("L = i + 1;", "L = (i + 2 < S) ? i + 2 : S;"),
    "max_over_first_key_only": ("for (long j = 0; j < L; ++j)\n        if (s[j] > m)", "for (long j = 0; j < 1; ++j)\n        if (s[j] > m)"),
    "partial_l_missing": ("lc += w;", "lc += 1.0;"),
    "partial_o_unweighted": ("oc[d] += w * widen(v,", "oc[d] += widen(v,"),
    "combine_l_unweighted": ("ls += lr[i] * w;", "ls += lr[i];"),
    "combine_o_unweighted": ("out_r[d] += orow[(size_t)i * D + d] * w;", "out_r[d] += orow[(size_t)i * D + d];"),
    "combine_all_empty_not_handled": ("if (ms == -INFINITY) {\n            lse[r] = -INFINITY;\n            continue;\n        }", ""),
    "empty_lse_zero": ("*lse = -INFINITY;\n        return;", "*lse = 0.0;\n        return;"),
    "bf16_low_bits_kept": ("<< 16;", "<< 15;"),
}


def _build_mutant(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation {name}: pattern not found"
    src = tmp_path / f"{name}.c"
    src.write_text(text.replace(old, new))
    lib = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-pthread",
                    str(src), "-o", str(lib), "-lm"], check=True)
    return str(lib)


def _bf16_pin():
    """bf16 inputs widen exactly: a bf16 tensor and its float32 copy give identical results."""
    import numpy as np
    import torch
    g = torch.Generator().manual_seed(5)
    q = torch.randn(1, 2, 8, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 1, 9, 8, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 1, 9, 8, generator=g).to(torch.bfloat16)
    a = oracle.decode(q, k, v, 0.5)
    b = oracle.decode(q.float(), k.float(), v.float(), 0.5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bf16_widening_is_exact():
    _bf16_pin()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(tmp_path, monkeypatch, name):
    old, new = MUTATIONS[name]
    path = _build_mutant(tmp_path, name, old, new)
    real = oracle.lib()
    mutant = ctypes.CDLL(path)
    for fn in ("oracle_decode", "oracle_prefill_causal", "oracle_decode_partials", "oracle_combine"):
        getattr(mutant, fn).argtypes = getattr(real, fn).argtypes
        getattr(mutant, fn).restype = getattr(real, fn).restype
    monkeypatch.setattr(oracle, "_lib", mutant)
    caught = []
    for pin in oracle_pins.ALL_PINS + [_bf16_pin]:
        try:
            pin()
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutation {name}"


# Mistakes planted in the paged oracle (a Python function): the mutated source
# is compiled into a copy of the function, swapped in, and every pin is run.
PY_MUTATIONS = {
    "page_rows_offset": ("kc[b, :, pg * page:(pg + 1) * page] = kp[table[b, pg]]",
                         "kc[b, :, pg * page:(pg + 1) * page] = kp[table[b, max(pg - 1, 0)]]"),
    "table_transposed": ("kp[table[b, pg]]", "kp[table[pg % B, b % P]]"),
    "last_page_dropped": ("npg = (int(lens[b]) + page - 1) // page", "npg = int(lens[b]) // page"),
    "v_from_k_pages": ("vc[b, :, pg * page:(pg + 1) * page] = vp[table[b, pg]]",
                       "vc[b, :, pg * page:(pg + 1) * page] = kp[table[b, pg]]"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTATIONS))
def test_paged_mutation_is_caught(monkeypatch, name):
    import inspect
    import textwrap
    old, new = PY_MUTATIONS[name]
    src = textwrap.dedent(inspect.getsource(oracle.decode_paged))
    assert src.count(old) >= 1, f"mutation {name}: pattern not found"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    monkeypatch.setattr(oracle, "decode_paged", ns["decode_paged"])
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutation {name}"


PI_MUTATIONS = {
    "window_excludes_newest": ("keys = set(range(max(0, i - window), i + 1))",
                               "keys = set(range(max(0, i - window), i))"),
    "window_one_short": ("keys = set(range(max(0, i - window), i + 1))",
                         "keys = set(range(max(0, i - window + 1), i + 1))"),
    "skips_from_window_start": ("j = i - period\n", "j = max(0, i - window) - period\n"),
    "skip_step_doubled": ("        j -= period", "        j -= 2 * period"),
}


@pytest.mark.parametrize("name", sorted(PI_MUTATIONS))
def test_pi_mutation_is_caught(monkeypatch, name):
    import inspect
    import textwrap
    old, new = PI_MUTATIONS[name]
    src = textwrap.dedent(inspect.getsource(oracle.pi_key_set))
    assert src.count(old) >= 1, f"mutation {name}: pattern not found"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    monkeypatch.setattr(oracle, "pi_key_set", ns["pi_key_set"])
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutation {name}"


VARLEN_MUTATIONS = {
    "starts_one_token_early": ("a, e = cu[s], cu[s + 1]", "a, e = max(cu[s] - 1, 0), cu[s + 1]"),
    "kv_heads_not_transposed": ("ks = np.ascontiguousarray(ka[a:e].transpose(1, 0, 2))[None]",
                                "ks = np.ascontiguousarray(ka[a:e].reshape(Hkv, e - a, D))[None]"),
    "lse_rows_swapped": ("lse[:, a:e] = l.reshape(H, e - a)", "lse[:, a:e] = l.reshape(e - a, H).T"),
    "output_not_transposed_back": ("out[a:e] = o.reshape(H, e - a, D).transpose(1, 0, 2)",
                                   "out[a:e] = o.reshape(e - a, H, D)"),
}


@pytest.mark.parametrize("name", sorted(VARLEN_MUTATIONS))
def test_varlen_prefill_mutation_is_caught(monkeypatch, name):
    import inspect
    import textwrap
    old, new = VARLEN_MUTATIONS[name]
    src = textwrap.dedent(inspect.getsource(oracle.prefill_causal_varlen))
    assert src.count(old) >= 1, f"mutation {name}: pattern not found"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    monkeypatch.setattr(oracle, "prefill_causal_varlen", ns["prefill_causal_varlen"])
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutation {name}"


FP8_MUTATIONS = {
    ("e2m1_to_float", "bias_2"): ("np.exp2(e - 1.0)", "np.exp2(e - 2.0)"),
    ("e2m1_to_float", "subnormal_as_normal"): ("np.where(e == 0, m / 2.0,", "np.where(e == 0, (1.0 + m / 2.0) * 0.5,"),
    ("nvfp4_dequantize", "nibbles_swapped"): ("np.stack([lo, hi], axis=-1)", "np.stack([hi, lo], axis=-1)"),
    ("nvfp4_dequantize", "block_of_32"): ("np.repeat(e4m3_to_float(bs), 16, axis=-1)",
                                          "np.repeat(e4m3_to_float(bs[..., ::2]), 32, axis=-1)"),
    ("nvfp4_dequantize", "block_scale_dropped"): ("vals = vals * np.repeat(e4m3_to_float(bs), 16, axis=-1)", "pass"),
    ("decode_nvfp4", "v_factor_dropped"): ("vd = nvfp4_dequantize(v4, v_bs, vf.reshape(B, Hkv, 1, 1))",
                                           "vd = nvfp4_dequantize(v4, v_bs, 1.0)"),
    ("e4m3_to_float", "bias_8"): ("np.exp2(e - 7.0)", "np.exp2(e - 8.0)"),
    ("e4m3_to_float", "subnormal_as_normal"): ("m / 8.0 * 2.0 ** -6", "(1.0 + m / 8.0) * 2.0 ** -7"),
    ("e4m3_to_float", "sign_ignored"): ("return np.where(s == 1, -mag, mag)", "return mag"),
    ("decode_fp8", "v_scale_dropped"): ("vd = e4m3_to_float(vb) * vs.reshape(B, Hkv, 1, 1)", "vd = e4m3_to_float(vb)"),
    ("decode_fp8", "k_scale_per_wrong_unit"): ("kd = e4m3_to_float(kb) * ks.reshape(B, Hkv, 1, 1)",
                                               "kd = e4m3_to_float(kb) * ks[::-1].reshape(B, Hkv, 1, 1)"),
}


@pytest.mark.parametrize("key", sorted(FP8_MUTATIONS), ids=lambda k: "-".join(k))
def test_fp8_mutation_is_caught(monkeypatch, key):
    import inspect
    import textwrap
    fn_name, _ = key
    old, new = FP8_MUTATIONS[key]
    src = textwrap.dedent(inspect.getsource(getattr(oracle, fn_name)))
    assert src.count(old) >= 1, f"mutation {key}: pattern not found"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant {key}>", "exec"), ns)
    monkeypatch.setattr(oracle, fn_name, ns[fn_name])
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutation {key}"
