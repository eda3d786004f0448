"""The oracle's pins catch plausible mistakes (CPU).

Each case copies oracle/sdpa_oracle.c, plants one mistake in the copy (a
dropped term, a wrong index or sign, a swapped operand, a wrong constant),
builds it into a temporary library, points the oracle module at it, and
runs the pins that guard that part of the oracle: at least one must fail.
The unchanged copy, built the same way, must pass all of them, so a failure
comes from the planted mistake and not from the build.  The oracle source
itself is never modified.
"""
import subprocess

import pytest
import torch

from oracle import oracle
from tests import test_oracle_feature_pins as feature_pins
from tests import test_oracle_fp8_pins as fp8_pins
from tests import test_oracle_pins as pins


def _sdpa_pins():
    pins.test_definition_matches_torch_sdpa(torch.bfloat16, True)
    pins.test_definition_matches_torch_sdpa(torch.float16, False)
    pins.test_lse_matches_logsumexp()


def _mask_pins():
    for shape in sorted(pins._read_masks().keys()):
        pins.test_causal_mask_matches_golden(shape)
    _sdpa_pins()


def _rounding_pins():
    for case in pins._golden_rounding():
        pins.test_rounding_golden(case)
    pins.test_bf16_rtz_and_rtna_closed_forms()


def _widen_pins():
    pins.test_widen_all_patterns(oracle.BF16, torch.bfloat16)
    pins.test_widen_all_patterns(oracle.F16, torch.float16)
    fp8_pins.test_widen8_matches_torch_on_all_patterns()


def _recurrence_pins():
    for tile in (3, 16):
        pins.test_streaming_recurrence_equals_definition(tile)
    for parts in (2, 8, 13):
        pins.test_split_combine_equals_definition(parts)


def _feature_pins():
    for left, right in ((3, -1), (0, 2), (2, 5)):
        feature_pins.test_window_matches_torch_band_mask(left, right)
    feature_pins.test_saturated_scores_take_plus_minus_cap()
    feature_pins.test_alibi_geometric_weights_closed_form()
    feature_pins.test_sink_with_zero_query_closed_form()
    feature_pins.test_row_without_keys_reports_the_sink()


def _fp8_pins():
    fp8_pins.test_fp8_matches_torch_sdpa_on_dequantised_values(True)
    fp8_pins.test_k_factor_scales_the_scores_and_v_factor_the_output()


MUTANTS = {
    # mask and indexing
    "causal mask aligned top-left": ("const int64_t diag = i + (Sk - Sq);",
                                     "const int64_t diag = i;", _mask_pins),
    "causal bound off by one": ("if (p->causal && diag + 1 < limit) limit = diag + 1;",
                                "if (p->causal && diag < limit) limit = diag;", _mask_pins),
    "GQA heads interleaved": ("int32_t kvh = h / (p->Hq / p->Hkv);",
                              "int32_t kvh = h % p->Hkv;", _sdpa_pins),
    "every key read from the sequence's first page": (
        "p->block_table[(int64_t)b * p->bt_stride + j / p->bs]",
        "p->block_table[(int64_t)b * p->bt_stride]", _sdpa_pins),
    # scores, weights, output
    "tau dropped": ("double x = p->scale * acc;", "double x = acc;", _sdpa_pins),
    "values read from the key cache": (
        "o[c] += w * cache_at(p, p->v_cache, p->v_scale, b, j, kvh, c);",
        "o[c] += w * cache_at(p, p->k_cache, p->k_scale, b, j, kvh, c);", _sdpa_pins),
    "normalisation dropped": ("for (int32_t c = 0; c < d; ++c) o[c] /= den;",
                              "for (int32_t c = 0; c < d; ++c) o[c] /= 1.0;", _sdpa_pins),
    "log-sum-exp in base 2": ("if (lse) *lse = m + log(den);",
                              "if (lse) *lse = m + log2(den);", _sdpa_pins),
    "running max left out of the log-sum-exp": ("if (lse) *lse = m + log(den);",
                                                "if (lse) *lse = log(den);", _sdpa_pins),
    # the streaming recurrence and the split combine
    "streaming: accumulator not rescaled": ("for (int32_t c = 0; c < d; ++c) o[c] *= alpha;",
                                            "for (int32_t c = 0; c < d; ++c) o[c] *= 1.0;",
                                            _recurrence_pins),
    "streaming: denominator not rescaled": ("l = alpha * l + tsum;", "l = l + tsum;",
                                            _recurrence_pins),
    "split: parts left unnormalised": ("for (int32_t c = 0; c < d; ++c) po[c] /= den;",
                                       "for (int32_t c = 0; c < d; ++c) po[c] /= 1.0;",
                                       _recurrence_pins),
    "split: combined LSE without the reference max": ("if (lse) *lse = L + log(wsum);",
                                                      "if (lse) *lse = log(wsum);",
                                                      _recurrence_pins),
    # feature flags
    "window: left bound taken from the right width": (
        "if (p->win_left >= 0 && diag - p->win_left > lo) lo = diag - p->win_left;",
        "if (p->win_left >= 0 && diag - p->win_right > lo) lo = diag - p->win_right;",
        _feature_pins),
    "softcap: outer factor dropped": (
        "if (p->softcap > 0.0) x = p->softcap * tanh(x / p->softcap);",
        "if (p->softcap > 0.0) x = tanh(x / p->softcap);", _feature_pins),
    "ALiBi bias added instead of subtracted": (
        "if (p->alibi) x -= p->alibi[h] * fabs((double)(diag - j));",
        "if (p->alibi) x += p->alibi[h] * fabs((double)(diag - j));", _feature_pins),
    "sink left out of the denominator": ("double den = p->sinks ? exp(sink - m) : 0.0;",
                                         "double den = 0.0;", _feature_pins),
    # formats
    "fp16 exponent bias off by one": ("v = ldexp((double)(1024 + f), e - 15 - 10);",
                                      "v = ldexp((double)(1024 + f), e - 16 - 10);",
                                      _widen_pins),
    "bf16 subnormals scaled as normals": ("v = ldexp((double)f, -126 - 7);",
                                          "v = ldexp((double)f, -127 - 7);", _widen_pins),
    "E4M3 subnormal exponent": ("mag = ldexp((double)f / 8.0, -6);",
                                "mag = ldexp((double)f / 8.0, -7);", _widen_pins),
    "E4M3 sign ignored": ("return s ? -mag : mag;", "return mag;", _widen_pins),
    "fp8 K factor ignored": (
        "acc += qv[c] * cache_at(p, p->k_cache, p->k_scale, b, j, kvh, c);",
        "acc += qv[c] * cache_at(p, p->k_cache, 1.0, b, j, kvh, c);", _fp8_pins),
    # rounding
    "RTNA rounds ties to even": ("else if (mode == OR_RTNA) up = cmp_half >= 0;",
                                 "else if (mode == OR_RTNA) up = cmp_half > 0;", _rounding_pins),
    "RTNE rounds every tie up": ("up = cmp_half > 0 || (cmp_half == 0 && (kept & 1));",
                                 "up = cmp_half >= 0;", _rounding_pins),
    "RTZ overflows to infinity": ("if (mode == OR_RTZ) return (uint16_t)(sign | maxfin);",
                                  "if (0) return (uint16_t)(sign | maxfin);", _rounding_pins),
}


def _build_copy(tmp_path, old=None, new=None):
    with open(oracle._SRC) as f:
        src = f.read()
    if old is not None:
        assert old in src, old
        src = src.replace(old, new)
    c = tmp_path / "oracle_copy.c"
    c.write_text(src)
    so = tmp_path / "liboracle_copy.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                    "-ffp-contract=off", "-o", str(so), str(c), "-lm", "-lpthread"], check=True)
    return str(so)


def _use(monkeypatch, so):
    monkeypatch.setattr(oracle, "build", lambda force=False: so)
    monkeypatch.setattr(oracle, "_lib", None)


def test_unchanged_copy_passes_every_battery(tmp_path, monkeypatch):
    _use(monkeypatch, _build_copy(tmp_path))
    for battery in {id(m[2]): m[2] for m in MUTANTS.values()}.values():
        battery()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_the_planted_mistake(name, tmp_path, monkeypatch):
    old, new, battery = MUTANTS[name]
    _use(monkeypatch, _build_copy(tmp_path, old, new))
    with pytest.raises(AssertionError):
        battery()
