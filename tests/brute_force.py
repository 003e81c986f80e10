"""Pure-Python brute force for tiny shapes: an independent second statement of the op, used
only to pin the oracle.  It shares nothing with oracle/gqa_oracle.c: visible sets are built
as Python set intersections, the sink is literally appended to the logit list and sliced
out afterwards, and every sum is math.fsum.  Inputs are Python floats.

Pages: OpenVINO PR #37423 ("Sliding window", "smooth_softmax / head_sink"), tract PR #2645
("What changed"), onnx-light-cpu "Attention Kernel Design" ("Layouts and semantics",
"Scheduling, precision, and invariants").
"""
import math


def visible_set(past, curr, i, window, causal):
    total = past + curr
    q_abs = past + i
    keep = set(range(total))
    if causal:
        keep &= set(range(q_abs + 1))
    if window >= 0:
        keep &= set(range(q_abs - window + 1, total + 1))
    return keep


def attention(q, present_k, present_v, seqlens, B, Hq, Hkv, D, curr, window, causal, scale,
              softcap=0.0, sinks=None, keep=None, bias=None, Dv=None):
    """q[b][i][hq] -> list of D floats; present_k[b][h][j] -> list of D floats.
    sinks: None, or a list of Hq floats.  keep(b, hq, i, j) -> bool removes keys from the
    row (a boolean mask); bias(b, hq, i, j) -> float is added to the scaled score before
    the softcap (an additive mask).  present_v rows hold Dv floats (default D).  Returns
    out[b][i][hq] lists of Dv floats."""
    G = Hq // Hkv
    Dv = D if Dv is None else Dv
    out = []
    for b in range(B):
        ob = []
        for i in range(curr):
            oi = []
            for hq in range(Hq):
                h = hq // G
                keys = sorted(visible_set(seqlens[b], curr, i, window, causal))
                if keep is not None:
                    keys = [j for j in keys if keep(b, hq, i, j)]
                logits = []
                values = []
                for j in keys:
                    s = scale * math.fsum(a * c for a, c in zip(q[b][i][hq], present_k[b][h][j]))
                    if bias is not None:
                        s = s + bias(b, hq, i, j)
                    if softcap > 0:
                        s = softcap * math.tanh(s / softcap)
                    if s == -math.inf:
                        continue   # exp(-inf) = 0: the key carries no weight
                    logits.append(s)
                    values.append(present_v[b][h][j])
                if not values:
                    oi.append([0.0] * Dv)
                    continue
                if sinks is not None:
                    logits.append(sinks[hq])   # extra logit in the denominator ...
                m = max(logits)
                e = [math.exp(x - m) for x in logits]
                den = math.fsum(e)
                p = [x / den for x in e][: len(values)]   # ... and sliced out
                oi.append([math.fsum(p[t] * values[t][d] for t in range(len(values))) for d in range(Dv)])
            ob.append(oi)
        out.append(ob)
    return out
