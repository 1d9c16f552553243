"""SwiGLU expert and the exact combine, in float64 (oracle, test infrastructure).

Passages followed:
  * snackonai deep dive "FreeToken, or why your laptop was never the
    bottleneck", section "What It Actually Does": the merge of the GPU's and
    the CPU's partial sums is exact; nothing in the routed computation is
    approximated.
  * same page, section "The split policy itself" (closing note): hits and
    filled experts are evaluated as grouped work on the GPU; misses assigned
    to the CPU execute where their weights live.
  * ai.thesatyajit.com article, section "Decode: the one equation": the two
    partial sums are combined without approximation.

The pages do not write out the expert.  The expert is the SwiGLU feed-forward
of the Qwen3 / DeepSeek-V3 MoE families the workloads are shaped after:
  g = W_gate x,  u = W_up x,  h = silu(g) * u,  y = W_down h,
  silu(z) = z / (1 + exp(-z)),
and the layer output is out[t] = sum_j w[t, j] * y[t, j] summed over j = 0..k-1
in that order, plus the shared expert's y (gate 1.0) when the model has one.
A pair (t, j) whose slot map entry is -1 takes its y from the supplied CPU
partial sums instead.
"""
from __future__ import annotations

from collections import OrderedDict

import numpy as np

from .formats import activations_to_f64, parse_blob


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z), the SwiGLU gate of the expert (reading: the
    pages do not write the expert out; Qwen3 and DeepSeek-V3 experts are SwiGLU)."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def swiglu_expert(x: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """y = W_down (silu(W_gate x) * (W_up x)) for x [..., H] -> [..., H], float64."""
    x = np.asarray(x, dtype=np.float64)
    g = x @ w_gate.T
    u = x @ w_up.T
    return (silu(g) * u) @ w_down.T


def swiglu_expert_loops(x, w_gate, w_up, w_down):
    """The same expert with explicit loops, for small shapes only."""
    I, H = w_gate.shape
    h = []
    for i in range(I):
        g = 0.0
        u = 0.0
        for c in range(H):
            g += float(w_gate[i][c]) * float(x[c])
            u += float(w_up[i][c]) * float(x[c])
        h.append(g / (1.0 + np.exp(-g)) * u)
    y = []
    for r in range(H):
        acc = 0.0
        for i in range(I):
            acc += float(w_down[r][i]) * h[i]
        y.append(acc)
    return np.array(y)


def combine(topk_w: np.ndarray, y_gpu: np.ndarray, slot_map: np.ndarray,
            cpu_part: np.ndarray | None, shared_y: np.ndarray | None = None) -> np.ndarray:
    """out[t] = sum over j in order of w[t,j] * (y_gpu[t,j] if slot_map[t,j] >= 0 else cpu_part[t,j]).

    topk_w [T,k], y_gpu/cpu_part [T,k,H], slot_map [T,k]; shared_y [T,H] is
    added last.  Entries of the unused source are never read.
    """
    T, k = topk_w.shape
    H = y_gpu.shape[-1]
    out = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        acc = np.zeros(H, dtype=np.float64)
        for j in range(k):
            if slot_map[t, j] >= 0:
                v = y_gpu[t, j]
            else:
                if cpu_part is None:
                    raise ValueError("a pair is CPU-assigned but no CPU partial sums were supplied")
                v = cpu_part[t, j]
            acc = acc + float(topk_w[t, j]) * np.asarray(v, dtype=np.float64)
        if shared_y is not None:
            acc = acc + shared_y[t]
        out[t] = acc
    return out


class ExpertStore:
    """Reads experts from a host pool (arena + per-expert byte offsets) as float64 matrices."""

    def __init__(self, arena: np.ndarray, offsets: np.ndarray, wdtype: str, H: int, I: int,
                 blob_bytes: int, memo: int = 16):
        self.arena = arena
        self.offsets = np.asarray(offsets, dtype=np.uint64)
        self.wdtype, self.H, self.I, self.S = wdtype, H, I, int(blob_bytes)
        self._memo: OrderedDict = OrderedDict()
        self._n = memo

    def blob(self, f: int) -> np.ndarray:
        """The S bytes of flat id f in the pool (snackonai "The Architecture,
        Unpacked": a slot, like a pool entry, holds one complete expert)."""
        o = int(self.offsets[f])
        return self.arena[o:o + self.S]

    def weights(self, f: int):
        """(W_gate, W_up, W_down) of flat id f as float64, decoded exactly."""
        key = int(self.offsets[f])
        if key in self._memo:
            self._memo.move_to_end(key)
            return self._memo[key]
        w = parse_blob(self.blob(f), self.wdtype, self.H, self.I)
        self._memo[key] = w
        if len(self._memo) > self._n:
            self._memo.popitem(last=False)
        return w

    def expert(self, f: int, x: np.ndarray) -> np.ndarray:
        """The SwiGLU expert f applied to x [..., H] in float64."""
        return swiglu_expert(x, *self.weights(f))


def pair_outputs(store: ExpertStore, layer: int, E: int, x: np.ndarray, adtype: str,
                 topk_ids: np.ndarray, mask: np.ndarray | None = None) -> np.ndarray:
    """y[t, j] = expert (layer*E + ids[t,j]) applied to x[t]; pairs with mask False stay zero."""
    xf = activations_to_f64(x, adtype)
    T, k = topk_ids.shape
    y = np.zeros((T, k, store.H), dtype=np.float64)
    # one pass per expert, all of its tokens at once
    for e in sorted({int(v) for v in np.asarray(topk_ids).ravel()}):
        sel = [(t, j) for t in range(T) for j in range(k)
               if int(topk_ids[t, j]) == e and (mask is None or mask[t, j])]
        if not sel:
            continue
        ts = [t for t, _ in sel]
        ye = store.expert(layer * E + e, xf[ts])
        for n, (t, j) in enumerate(sel):
            y[t, j] = ye[n]
    return y


def shared_outputs(shared_blobs: np.ndarray, layer: int, wdtype: str, H: int, I: int,
                   blob_bytes: int, x: np.ndarray, adtype: str) -> np.ndarray:
    """The always-resident shared expert of `layer` applied to x (reading: the
    DeepSeek-V3 shape's shared expert; signalovernoise.tech and dev.to: only
    the routed experts leave the GPU), added last by the combine."""
    blob = shared_blobs[layer * blob_bytes:(layer + 1) * blob_bytes]
    return swiglu_expert(activations_to_f64(x, adtype), *parse_blob(blob, wdtype, H, I))


def relative_max_error(y: np.ndarray, y_ref: np.ndarray) -> float:
    """max |y - y_ref| / max |y_ref| (the tolerance metric for floating-point outputs)."""
    y_ref = np.asarray(y_ref, dtype=np.float64)
    den = float(np.max(np.abs(y_ref))) if y_ref.size else 0.0
    num = float(np.max(np.abs(np.asarray(y, dtype=np.float64) - y_ref))) if y_ref.size else 0.0
    return num / den if den > 0 else num
