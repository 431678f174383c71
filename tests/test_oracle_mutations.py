"""The oracle's pins must catch plausible mistakes.  Each mutant below is the
oracle with one mistake planted (a wrong rounding rule, a dropped term, a
swapped operand or index, an off-by-one block), installed in place of the
real function on the CPU; at least one of the pins of that function must then
fail.  Nothing here touches the GPU."""
import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

_real = {name: getattr(oracle, name) for name in (
    "quantize_rows", "gemm_s32", "gemm_s32_f64", "epilogue", "bf16_linear_f64", "quantize_qk_blocks",
    "norm_modulate_f64")}


def _widen(A):
    A = np.asarray(A)
    return oracle.bf16_bits_to_f32(A) if A.dtype == np.uint16 else A.astype(np.float32)


def _quant_mutant(scale_div=127.0, rounding="even", clamp=127, zero_scale=1.0):
    def q(A, dtype=None):
        x = _widen(A)
        amax = np.abs(x).max(axis=1)
        s = (amax / np.float32(scale_div)).astype(np.float32)
        zero = s == 0
        s = np.where(zero, np.float32(zero_scale), s).astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            v = (x / s[:, None]).astype(np.float32)
        if rounding == "even":
            c = np.rint(v)
        elif rounding == "half_up":
            c = np.floor(v + np.float32(0.5))
        else:
            c = np.trunc(v)
        c = np.nan_to_num(np.clip(c, -clamp, clamp))
        return c.astype(np.int8), s
    return q


def _gemm_mutant(kind):
    def g(Xq, Wq, rows=None):
        xq = np.asarray(Xq).astype(np.int64)
        wq = np.asarray(Wq).astype(np.int64)
        if rows is not None:
            xq = xq[np.asarray(rows)]
        if kind == "drop_last_k":
            xq, wq = xq[:, :-1], wq[:, :-1]
        if kind == "weights_reversed":
            wq = wq[::-1]
        acc = xq @ wq.T
        if kind == "wrap":
            return acc.astype(np.int32)      # silently wraps past INT32
        return acc.astype(np.int32)
    return g


def _epilogue_mutant(kind):
    real = _real["epilogue"]

    def e(acc, sx, sw, bias=None):
        if kind == "no_bias":
            return real(acc, sx, sw, None)
        if kind == "scales_swapped":
            n = min(len(sx), len(sw))
            return real(acc, np.resize(sw, len(sx)).astype(np.float32), np.resize(sx, len(sw)).astype(np.float32),
                        bias) if n else real(acc, sx, sw, bias)
        if kind == "scales_first":
            # acc * (sx * sw): the two scales multiplied first, in fp32
            acc = np.asarray(acc)
            s2 = (np.asarray(sx, np.float32)[:, None] * np.asarray(sw, np.float32)[None, :]).astype(np.float32)
            y32 = (acc.astype(np.float32) * s2).astype(np.float32)
            if bias is not None:
                y32 = (y32 + np.asarray(bias, np.float32)[None, :]).astype(np.float32)
            return y32, oracle.bf16_rne(y32)
        return real(acc, sx, sw, bias)
    return e


def _bf16_linear_mutant(kind):
    real = _real["bf16_linear_f64"]

    def f(X_bits, W_bits, bias=None, rows=None):
        if kind == "no_bias":
            return real(X_bits, W_bits, None, rows)
        if kind == "w_not_transposed" and W_bits.shape[0] == W_bits.shape[1]:
            return real(X_bits, np.ascontiguousarray(W_bits.T), bias, rows)
        if kind == "w_not_transposed":
            return real(X_bits, W_bits[::-1].copy(), bias, rows)
        return real(X_bits, W_bits, bias, rows)
    return f


def _qk_mutant(kind):
    real = _real["quantize_qk_blocks"]

    def f(X, block_tokens, layout="HND"):
        if kind == "block_off_by_one":
            return real(X, block_tokens + 1 if block_tokens < X.shape[2 if layout == "HND" else 1] else block_tokens,
                        layout)
        if kind == "layout_ignored":
            return real(X, block_tokens, "HND")
        return real(X, block_tokens, layout)
    return f


def _norm_mutant(kind):
    def f(X_bits, kind_, eps, scale=None, shift=None):
        x = oracle.bf16_bits_to_f32(np.ascontiguousarray(X_bits)).astype(np.float64)
        K = x.shape[1]
        mu = x.sum(axis=1) / K if kind_ == "layer" else np.zeros(x.shape[0])
        d = x - mu[:, None]
        if kind == "no_eps":
            r = 1.0 / np.sqrt((d * d).sum(axis=1) / K)
        elif kind == "no_centering":
            r = 1.0 / np.sqrt((x * x).sum(axis=1) / K + eps)
        else:
            r = 1.0 / np.sqrt((d * d).sum(axis=1) / K + eps)
        y = d * r[:, None]
        if scale is not None:
            y = y * (np.asarray(scale, dtype=np.float64)[None, :] if kind == "scale_not_plus_one"
                     else (1.0 + np.asarray(scale, dtype=np.float64))[None, :])
        if shift is not None:
            y = y + np.asarray(shift, dtype=np.float64)[None, :]
        return y, mu, r
    return f


QUANT_PINS = [lambda: pins.test_quant_lossless_power_of_two_scale(3), pins.test_quant_all_255_codes_brute_force,
              pins.test_quant_ties_round_half_to_even, pins.test_quant_zero_row_scale_one,
              pins.test_quant_invariants_random, pins.test_quant_single_element_rows]
GEMM_PINS = [pins.test_gemm_k1_all_code_pairs_brute_force, pins.test_gemm_hand_expanded,
             pins.test_gemm_identity_and_permutation, pins.test_gemm_all_127_row_closed_form,
             pins.test_gemm_matches_numpy_int64_matmul, pins.test_gemm_int32_limit,
             pins.test_gemm_f64_path_equals_scalar_path_large_sums]
EPI_PINS = [pins.test_epilogue_zero_acc_gives_bias, pins.test_epilogue_exact_powers_of_two,
            pins.test_epilogue_indices_against_float64, pins.test_linear_zero_row_outputs_bias,
            pins.test_epilogue_rounding_order]
BF16_PINS = [pins.test_bf16_linear_brute_force, pins.test_bf16_linear_identity_and_roles,
             pins.test_bf16_linear_closed_form_and_tolerance]
QK_PINS = [pins.test_qk_blocks_brute_force, pins.test_qk_blocks_layouts_agree, pins.test_qk_blocks_special_block_sizes,
           pins.test_qk_blocks_are_independent_and_saturate]
NORM_PINS = [pins.test_norm_brute_force, pins.test_norm_closed_forms, pins.test_norm_invariances_and_modulation]

MUTANTS = [
    ("quantize_rows", "round half up", _quant_mutant(rounding="half_up"), QUANT_PINS),
    ("quantize_rows", "truncate", _quant_mutant(rounding="trunc"), QUANT_PINS),
    ("quantize_rows", "scale amax/128", _quant_mutant(scale_div=128.0), QUANT_PINS),
    ("quantize_rows", "clamp to 126", _quant_mutant(clamp=126), QUANT_PINS),
    ("quantize_rows", "zero row scale 0", _quant_mutant(zero_scale=0.0), QUANT_PINS),
    ("gemm_s32", "last k term dropped", _gemm_mutant("drop_last_k"), GEMM_PINS),
    ("gemm_s32", "weight rows reversed", _gemm_mutant("weights_reversed"), GEMM_PINS),
    ("gemm_s32", "INT32 overflow unreported", _gemm_mutant("wrap"), GEMM_PINS),
    ("gemm_s32_f64", "last k term dropped", _gemm_mutant("drop_last_k"), GEMM_PINS),
    ("epilogue", "bias dropped", _epilogue_mutant("no_bias"), EPI_PINS),
    ("epilogue", "row and column scales swapped", _epilogue_mutant("scales_swapped"), EPI_PINS),
    ("epilogue", "scales multiplied together first", _epilogue_mutant("scales_first"), EPI_PINS),
    ("bf16_linear_f64", "bias dropped", _bf16_linear_mutant("no_bias"), BF16_PINS),
    ("bf16_linear_f64", "W not transposed", _bf16_linear_mutant("w_not_transposed"), BF16_PINS),
    ("quantize_qk_blocks", "block one token too long", _qk_mutant("block_off_by_one"), QK_PINS),
    ("quantize_qk_blocks", "token-major layout read as head-major", _qk_mutant("layout_ignored"), QK_PINS),
    ("norm_modulate_f64", "eps dropped", _norm_mutant("no_eps"), NORM_PINS),
    ("norm_modulate_f64", "LayerNorm variance not centred", _norm_mutant("no_centering"), NORM_PINS),
    ("norm_modulate_f64", "scale instead of 1 + scale", _norm_mutant("scale_not_plus_one"), NORM_PINS),
]


@pytest.mark.parametrize("name,what,mutant,pin_list", MUTANTS, ids=["%s: %s" % (m[0], m[1]) for m in MUTANTS])
def test_pins_catch_planted_mistake(monkeypatch, name, what, mutant, pin_list):
    monkeypatch.setattr(oracle, name, mutant)
    caught = []
    for pin in pin_list:
        try:
            pin()
        except (Exception, pytest.fail.Exception):   # an assertion, pytest.raises failing, or the
            caught.append(getattr(pin, "__name__", "pin"))   # mutant's output breaking the pin's arithmetic
    assert caught, "no pin of %s caught: %s" % (name, what)


def test_unmutated_oracle_passes_the_same_pins():
    """The control: with the real functions every pin used above passes."""
    for pin in QUANT_PINS + GEMM_PINS + EPI_PINS + BF16_PINS + QK_PINS + NORM_PINS:
        pin()
