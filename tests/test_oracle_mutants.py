"""Plant plausible mistakes in the oracle (on the CPU, in throw-away builds) and check that
the pins catch every one: a dropped term, a wrong sign, index or operand, an off-by-one in
the causal limit, a wrong exponent bias. A mistake no pin catches fails this test."""
import ctypes
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.c")

MUTANTS = {
    "scores_skip_rope_dims": ("acc += q[d] * table[row[d]];",
                              "acc += (d < 512 ? q[d] * table[row[d]] : 0.0);"),
    "causal_off_by_one": ("seq_lens[b] - n_q + j + 1;", "seq_lens[b] - n_q + j;"),
    "value_from_wrong_dims": ("out[d] += w * table[row[d]];", "out[d] += w * table[row[d + 64]];"),
    "softmax_sign": ("double w = exp(scores[n - lo] - l);", "double w = exp(l - scores[n - lo]);"),
    "e4m3_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3_subnormal_scale": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "page_offset": ("(n % page_size)) * ORACLE_D", "(n / page_size)) * ORACLE_D"),
    "q_layout_transposed": ("(((int64_t)b * n_q + j) * H + h)", "(((int64_t)b * H + h) * n_q + j)"),
    "lse_missing_max": ("double l = m + log(sum);\n  for (int64_t n = lo;",
                        "double l = log(sum);\n  for (int64_t n = lo;"),
    "merge_lse_missing_max": ("double l = m + log(sum);\n    for (int s = 0;",
                              "double l = log(sum);\n    for (int s = 0;"),
    "sm_scale_dropped": ("scores[n - lo] = sm_scale * acc;", "scores[n - lo] = acc;"),
    "bf16_shift": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    "merge_weight_no_norm": ("double w = exp(part_lse[(int64_t)s * R + r] - l);",
                             "double w = exp(part_lse[(int64_t)s * R + r] - m);"),
    "kv_scale_dropped": ("table[c] = oracle_e4m3_value((uint8_t)c) * kv_scale;",
                         "table[c] = oracle_e4m3_value((uint8_t)c);"),
    "e4m3_nan_code": ("if (e == 0xF && m == 0x7) return NAN;", "if (e == 0xF && m == 0x6) return NAN;"),
    "encode_ties_up": ("(err == best_err && (c & 1) == 0 && (best & 1) == 1)", "(err == best_err)"),
    "encode_drops_sign": ("const uint8_t sign = signbit(v) ? 0x80 : 0x00;",
                          "const uint8_t sign = v < 0 ? 0x80 : 0x00;"),
    "encode_no_saturation": ("if (a > 448.0) a = 448.0;", ""),
    "append_scale_not_inverted": ("const float prod = x * inv;", "const float prod = x * kv_scale;"),
    "append_row_offset": ("pool[s * ORACLE_D + d] =", "pool[(s + 1) * ORACLE_D + d - ORACLE_D * (s == pool_rows - 1)] ="),
}


def _build_mutant(name, old, new, tmp):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(tmp, f"lib{name}.so")
    inc = os.path.dirname(SRC)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", f"-I{inc}", "-o", so,
                    path, "-lm"], check=True)
    return oracle.bind(ctypes.CDLL(so))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    with tempfile.TemporaryDirectory() as tmp:
        lib = _build_mutant(name, old, new, tmp)
        prev = oracle.use_library(lib)
        caught = []
        try:
            for pin in oracle_pins.ALL_PINS:
                try:
                    pin(oracle)
                except (AssertionError, ValueError):
                    caught.append(pin.__name__)
        finally:
            oracle.use_library(prev)
    assert caught, f"no pin caught mutant {name}"


# Mistakes planted in the oracle's Python-level functions (top-k renormalisation).
PY_MUTANTS = {
    "topk_drops_ties": ("keep = p[r] >= pivot", "keep = p[r] > pivot"),
    "topk_off_by_one_pivot": ("pivot = np.sort(p[r])[V - k]", "pivot = np.sort(p[r])[V - k - 1]"),
    "topk_renorm_by_row_sum": ("out[r, keep] = p[r, keep] / p[r, keep].sum()",
                               "out[r, keep] = p[r, keep] / p[r].sum()"),
    "topk_keep_all_at_v_minus_1": ("if k <= 0 or k >= V:", "if k <= 0 or k >= V - 1:"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_py_mutant_is_caught(name):
    import inspect
    import types
    old, new = PY_MUTANTS[name]
    src = inspect.getsource(oracle.top_k_renorm_prob)
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    ns = dict(vars(oracle))
    exec(src.replace(old, new), ns)
    shim = types.SimpleNamespace(top_k_renorm_prob=ns["top_k_renorm_prob"])
    with pytest.raises(AssertionError):
        oracle_pins.pin_top_k_renorm(shim)


# Mistakes planted in the MHA-form prefill oracle.
MHA_MUTANTS = {
    "mha_drops_rope": ("K = np.concatenate([c @ W[:, h, :128], r], axis=1)",
                       "K = np.concatenate([c @ W[:, h, :128], 0 * r], axis=1)"),
    "mha_uk_uv_swapped": ("V = c @ W[:, h, 128:]", "V = c @ W[:, h, :128]"),
    "mha_causal_off_by_one": ("<= (L - T + ts)[:, None]", "< (L - T + ts)[:, None]"),
    "mha_head_of_weights": ("K = np.concatenate([c @ W[:, h, :128], r], axis=1)",
                            "K = np.concatenate([c @ W[:, 0, :128], r], axis=1)"),
    "mha_no_scale": ("s = float(cache.sm_scale) * (qf[ts, h, :] @ K.T)", "s = qf[ts, h, :] @ K.T"),
}


@pytest.mark.parametrize("name", sorted(MHA_MUTANTS))
def test_mha_mutant_is_caught(name):
    import inspect
    import types
    old, new = MHA_MUTANTS[name]
    src = inspect.getsource(oracle.mha_prefill_rows)
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    ns = dict(vars(oracle))
    exec(src.replace(old, new), ns)
    shim = types.SimpleNamespace(**{k: getattr(oracle, k) for k in ("attention", "e4m3_value")},
                                 mha_prefill_rows=ns["mha_prefill_rows"])
    caught = []
    for pin in (oracle_pins.pin_mha_absorbed_identity, oracle_pins.pin_mha_zero_query,
                oracle_pins.pin_mha_sdpa):
        try:
            pin(shim)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
