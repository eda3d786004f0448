"""The algorithmic work bench.py divides by (CPU): the visible (query, key)
pair count behind every prefill TFLOP/s figure and the K/V + Q/O byte count
behind every decode GB/s figure.  Pinned against the hand-worked causal
masks of tests/golden, brute-force enumeration of the mask definition
("gfx942 unified attention, from the math up", sec. 4: bottom-right
alignment, key j visible to row i iff j <= i + Sk - Sq; the sliding window
keeps diag - left <= j <= diag + right), closed forms, and the sizes of the
decode tensors as built."""
import os

import numpy as np
import pytest
import torch

import attn_inputs
import bench

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def brute_pairs(sq, sk, causal, window=(-1, -1)):
    n = 0
    for i in range(sq):
        diag = i + sk - sq
        for j in range(sk):
            if causal and j > diag:
                continue
            if window[0] >= 0 and j < diag - window[0]:
                continue
            if window[1] >= 0 and j > diag + window[1]:
                continue
            n += 1
    return n


def test_pairs_match_the_hand_worked_masks():
    shapes = {}
    with open(os.path.join(GOLDEN, "causal_masks.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            head, keys = line.split(":")
            sq, sk, _ = (int(x) for x in head.split())
            k = keys.split()
            shapes[(sq, sk)] = shapes.get((sq, sk), 0) + (0 if k == ["-"] else len(k))
    assert shapes
    for (sq, sk), n in shapes.items():
        assert bench.visible_pairs([sq], [sk], True) == n, (sq, sk)


@pytest.mark.parametrize("seed", range(6))
def test_pairs_match_brute_force(seed):
    rng = np.random.default_rng(seed)
    for _ in range(40):
        n = int(rng.integers(1, 4))
        q = [int(x) for x in rng.integers(0, 30, size=n)]
        k = [int(x) for x in rng.integers(0, 40, size=n)]
        causal = bool(rng.integers(2))
        window = (int(rng.integers(-1, 12)), int(rng.integers(-1, 6)))
        want = sum(brute_pairs(a, b, causal, window) for a, b in zip(q, k))
        assert bench.visible_pairs(q, k, causal, window) == want, (q, k, causal, window)


def test_pairs_closed_forms():
    assert bench.visible_pairs([2048], [2048], True) == 2048 * 2049 // 2
    assert bench.visible_pairs([300], [700], False) == 300 * 700
    # bottom-right causal with Sk >= Sq: row i sees Sk - Sq + i + 1 keys
    assert bench.visible_pairs([100], [612], True) == sum(512 + i + 1 for i in range(100))
    # a left window of w over a square causal mask: min(i, w) + 1 keys per row
    assert bench.visible_pairs([500], [500], True, (64, -1)) == sum(min(i, 64) + 1
                                                                   for i in range(500))


def test_headline_prefill_flops():
    prob = attn_inputs.workload("prefill_causal_bf16_gqa_s2048")
    # 4 d FLOPs per visible pair per query head: S = QK^T and O = PV
    assert bench.prefill_flops(prob) == 4.0 * 128 * 32 * (2048 * 2049 // 2) == 34376515584.0


def test_headline_decode_bytes_are_the_tensors_read_and_written():
    prob = attn_inputs.workload("decode_bf16_b64_paged16")
    d, hkv, hq, b = prob.head_size, prob.num_kv_heads, prob.num_q_heads, prob.num_seqs
    kv_rows = int(np.sum(prob.seq_lens.numpy()))
    assert kv_rows == sum(prob.kv_lens)
    want = 2 * kv_rows * hkv * d * 2 + prob.q.numel() * 2 + b * hq * d * 2
    assert bench.decode_bytes(prob) == float(want)
    # a left window of w reads the last w + 1 keys of each sequence
    w = 1024
    keys = sum(min(int(s), w + 1) for s in prob.seq_lens.numpy())
    assert bench.decode_bytes(prob, (w, -1)) == float(2 * keys * hkv * d * 2 + 2 * b * hq * d * 2)


def test_fp8_decode_bytes_count_one_byte_per_cached_element():
    prob = attn_inputs.workload("decode_bf16_b64_paged16", kv_dtype=torch.float8_e4m3fn)
    assert prob.kv_fp8
    kv_rows = sum(prob.kv_lens)
    d, hkv, hq, b = prob.head_size, prob.num_kv_heads, prob.num_q_heads, prob.num_seqs
    assert bench.decode_bytes(prob) == float(2 * kv_rows * hkv * d + 2 * b * hq * d * 2)


def test_code_hash_ignores_comments_and_layout_but_not_code():
    """The traffic figures in bench.py are tied to the kernel source through
    this hash: comment and white-space edits keep them, code edits drop them."""
    a = "int f(int x) {\n  return x + 1;  // one\n}\n/* block\n comment */\n"
    b = "int f(int x){return x+1;}   // other words\n"
    c = "int f(int x) { return x + 2; }\n"
    assert bench.code_hash(a) == bench.code_hash(b)
    assert bench.code_hash(a) != bench.code_hash(c)


def test_clock_samples_are_kept_from_timed_spans_and_summarised():
    """The clock record: only samples inside the timed wall-time spans count;
    the SM clock is their median, the maximum the highest seen, and a throttle
    reason is reported when any sample shows it active."""
    s = bench.ClockSampler(0)
    # nvidia-smi lines: sm, max sm, power, active mask, hw, hw thermal, sw thermal, sw power cap
    s.samples = [
        (1.0, "1000, 2070, 300.0, 0x1, Not Active, Not Active, Not Active, Not Active"),   # idle, before
        (2.0, "2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
        (2.5, "2070, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active"),
        (3.0, "2040, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active"),
        (9.0, "300, 2070, 100.0, 0x1, Active, Not Active, Not Active, Not Active"),       # after
        (9.5, "garbage line"),
    ]
    inside = s.parsed(1.5, 3.5)
    assert [x[0] for x in inside] == [2070.0, 2070.0, 2040.0]
    c = bench.clock_summary(inside, "timed")
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                 "samples": 3, "window": "timed"}
    # pooled spans, as the line's record pools the step with the configuration set
    pooled = bench.clock_summary(s.parsed(1.5, 2.2) + s.parsed(8.5, 9.9), "two spans")
    assert pooled["samples"] == 2 and pooled["reasons"] == ["hw_slowdown"]
    assert pooled["sm_mhz"] == (2070.0 + 300.0) / 2
    # no sample inside: the whole run is summarised and labelled so
    assert s.summary(4.0, 5.0)["window"] == "whole run"
    assert bench.clock_summary([], "timed")["samples"] == 0
