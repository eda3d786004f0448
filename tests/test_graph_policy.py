"""The graph-replay policy of "gfx942 unified attention, from the math up",
sec. 9 (host logic, no GPU): decode and prefill of at most 768 query rows are
graphed, longer prefill and feature-flagged calls are not; and the cache key
changes with every pointer, shape and scalar that a recorded graph would bake
in."""
import torch

import attention_forward_sdpa_gb300 as attn
from attention_forward_sdpa_gb300 import graphs


def test_policy_thresholds():
    assert graphs.should_graph(1)          # decode
    assert graphs.should_graph(128)
    assert graphs.should_graph(768)        # the threshold itself is graphed
    assert not graphs.should_graph(769)
    assert not graphs.should_graph(8192)
    assert not graphs.should_graph(0)      # nothing to run


def test_feature_flagged_calls_are_not_graphed():
    assert not graphs.should_graph(1, True)
    assert not graphs.should_graph(128, True)
    assert not attn.has_features()
    assert attn.has_features(window=(128, -1))
    assert attn.has_features(softcap=30.0)
    assert attn.has_features(alibi_slopes=torch.zeros(4))
    assert attn.has_features(sinks=torch.zeros(4))


def test_cache_key_sees_pointers_shapes_and_scalars():
    a = torch.zeros(4, 8)
    b = torch.zeros(4, 8)
    k1 = graphs._key("decode", (a, None), (1, 0.5))
    assert k1 == graphs._key("decode", (a, None), (1, 0.5))
    assert k1 != graphs._key("decode", (b, None), (1, 0.5))            # another tensor
    assert k1 != graphs._key("decode", (a.view(8, 4), None), (1, 0.5))  # another shape
    assert k1 != graphs._key("decode", (a, None), (2, 0.5))            # another scalar
    assert k1 != graphs._key("prefill", (a, None), (1, 0.5))           # another entry point
