"""CUDA-graph replay for launch-bound calls.

The dispatcher of "gfx942 unified attention, from the math up" (sec. 9)
replays decode steps and short prefills from a captured graph and runs long
prefills eagerly: a decode step (one query row per sequence) or a prefill of
at most 768 query rows is dominated by launch and host time, a long prefill
is not.  Feature-flagged calls (sliding window, softcap, ALiBi, sinks) are
never graphed, as there.  A call made while the caller's stream is already
being captured is simply recorded into the caller's graph instead.

A graph bakes in every pointer, size and scalar of the call it recorded, so
the cache is keyed on all of them: replaying a key runs the same kernels on
the same tensors, reading whatever values those tensors hold at replay time.
The caller keeps the tensors alive (the cache holds references to them).
"""
from __future__ import annotations

import torch

from . import attn_decode_workspace_size, attn_fwd_decode, attn_fwd_prefill, has_features

GRAPH_MAX_SEQLEN_Q = 768   # the pages' threshold: graph at or below, eager above


def should_graph(max_seqlen_q: int, featured: bool = False) -> bool:
    """The replay policy: decode (max_seqlen_q == 1) and short prefill
    (max_seqlen_q <= 768) are graphed; longer prefill and feature-flagged
    calls are not."""
    return not featured and 1 <= int(max_seqlen_q) <= GRAPH_MAX_SEQLEN_Q


def _key(name, tensors, scalars):
    parts = [name]
    for t in tensors:
        if t is None:
            parts.append(None)
        else:
            parts.append((t.data_ptr(), tuple(t.shape), tuple(t.stride()), str(t.dtype),
                          t.device.index))
    parts.extend(scalars)
    return tuple(parts)


class GraphCache:
    """Captures each distinct call once and replays it afterwards."""

    def __init__(self):
        self._graphs: dict = {}
        self._capture_stream = None
        self.captures = 0
        self.replays = 0

    def __len__(self) -> int:
        return len(self._graphs)

    def clear(self) -> None:
        self._graphs.clear()

    def run(self, key, tensors, fn) -> None:
        """fn(stream) enqueues the call on `stream`; it is captured on first use
        of `key` and replayed on the current stream from then on.  The
        caller makes the tensors' device current."""
        cur = torch.cuda.current_stream()
        if torch.cuda.is_current_stream_capturing():
            fn(cur)                      # the caller's own capture records it
            return
        entry = self._graphs.get(key)
        if entry is None:
            if self._capture_stream is None:
                self._capture_stream = torch.cuda.Stream()
            cap = self._capture_stream
            cap.wait_stream(cur)
            with torch.cuda.stream(cap):
                fn(cap)                  # first call eagerly: one-time setup stays out of the graph
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                fn(cap)
            cur.wait_stream(cap)
            entry = (g, tuple(tensors))  # keep the tensors the graph points at alive
            self._graphs[key] = entry
            self.captures += 1
            return                       # the eager call above already produced the result
        entry[0].replay()
        self.replays += 1


_default = GraphCache()


def default_cache() -> GraphCache:
    return _default


def decode(out, q, k_cache, v_cache, block_table, seq_lens, *, max_seqlen_k: int, scale: float,
           num_splits: int, workspace, rounding: int = 0, lse=None, cache: GraphCache | None = None,
           **features) -> bool:
    """attn_fwd_decode through the replay cache (decode is graphed unless it
    carries feature flags, which run eagerly).  The workspace must be
    supplied (a graph cannot allocate).  Returns True when the call went
    through the cache."""
    if workspace is None:
        raise ValueError("graphed decode needs a caller workspace of "
                         "attn_decode_workspace_size(...) bytes")
    if not should_graph(1, has_features(**features)):
        attn_fwd_decode(out, q, k_cache, v_cache, block_table, seq_lens,
                        max_seqlen_k=max_seqlen_k, scale=scale, num_splits=num_splits,
                        workspace=workspace, rounding=rounding, lse=lse, **features)
        return False
    cache = _default if cache is None else cache
    tensors = (out, q, k_cache, v_cache, block_table, seq_lens, workspace, lse)
    key = _key("decode", tensors, (int(max_seqlen_k), float(scale), int(num_splits),
                                   int(rounding)))

    def fn(stream):
        attn_fwd_decode(out, q, k_cache, v_cache, block_table, seq_lens,
                        max_seqlen_k=max_seqlen_k, scale=scale, num_splits=num_splits,
                        workspace=workspace, rounding=rounding, lse=lse, stream=stream)

    with torch.cuda.device(q.device):
        cache.run(key, tensors, fn)
    return True


def prefill(out, q, k_cache, v_cache, block_table, query_start_loc, seq_lens, *,
            max_seqlen_q: int, max_seqlen_k: int, scale: float, causal: bool, rounding: int = 0,
            lse=None, cache: GraphCache | None = None, **features) -> bool:
    """attn_fwd_prefill, replayed from a graph when the policy says so.
    Returns True when the call went through the cache."""
    def fn(stream):
        attn_fwd_prefill(out, q, k_cache, v_cache, block_table, query_start_loc, seq_lens,
                         max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k, scale=scale,
                         causal=causal, rounding=rounding, lse=lse, stream=stream, **features)

    if not should_graph(max_seqlen_q, has_features(**features)):
        fn(None)                         # the query device's current stream
        return False
    cache = _default if cache is None else cache
    tensors = (out, q, k_cache, v_cache, block_table, query_start_loc, seq_lens, lse)
    key = _key("prefill", tensors, (int(max_seqlen_q), int(max_seqlen_k), float(scale),
                                    bool(causal), int(rounding)))
    with torch.cuda.device(q.device):
        cache.run(key, tensors, fn)
    return True


__all__ = ["GRAPH_MAX_SEQLEN_Q", "should_graph", "GraphCache", "default_cache", "decode",
           "prefill", "attn_decode_workspace_size"]
