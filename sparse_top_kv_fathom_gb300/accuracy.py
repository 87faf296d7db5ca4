"""Synthetic accuracy of the selection: attention error and top-k recall against the budget.

For one layer of a synthetic workload (keys, values and queries from `synth`), every
(budget B, GQA reading) pair runs the library's own decode step -- allocation, bit-plane
scan, top-k and sparse attention on the GPU -- and is compared with two references
computed here in plain torch on the original 16-bit K/V:

* recall: the share of the exact top-k keys (by the exact logits q.K, summed over the group
  for the "sum" reading, per head for "per_head", the max over the group's heads for "max")
  that the step selected;
* error: ||o - o_dense|| / ||o_dense|| per query head (mean over heads), o_dense being full
  softmax attention over all n keys; the same with attention's keys read back from the 4-bit
  index (the unified store) instead of the 16-bit K; and for the exact top-k's attention
  ("exact-k"), the floor any k-key selection reaches;
* error against the exact top-k: the same norm with the exact top-k's attention output as the
  reference, which isolates how much of it the selection (and the 4-bit keys) give up.  On
  these synthetic keys attention is spread thin over all n keys, so errors against dense
  attention are large for any k-key selection.

The pages measure this on real models and tasks (needle-in-a-haystack, recall against the
fixed-channel index); those are not available, so this is the synthetic analogue.  Run:
    python -m sparse_top_kv_fathom_gb300.accuracy [--workload qwen_layer] [--n N]
"""
import argparse
import json
import math

import torch

from . import api as F
from . import synth


def dense_attention(q, K, V, group):
    """softmax(q K^T / sqrt(128)) V over all keys, fp32: q [rows*group][128], K/V [rows][n][128]."""
    rows, n, d = K.shape
    qf = q.float().view(rows, group, d)
    logits = torch.einsum("rgd,rnd->rgn", qf, K.float()) / math.sqrt(d)
    return torch.einsum("rgn,rnd->rgd", torch.softmax(logits, -1), V.float()).reshape(rows * group, d)


def exact_sets(q, K, group, k, mode):
    """Exact top-k indices [sets][k] (ties to the lower index) under a GQA reading."""
    rows, n, d = K.shape
    logits = torch.einsum("rgd,rnd->rgn", q.float().view(rows, group, d), K.float())
    if mode == "sum":
        s = logits.sum(1)
    elif mode == "max":
        s = logits.max(1).values
    else:
        s = logits.reshape(rows * group, n)
    return F.topk(s.contiguous(), k)


def recall(sel, ref):
    """Mean over sets of |sel & ref| / |ref|."""
    hits = []
    for a, b in zip(sel.cpu().tolist(), ref.cpu().tolist()):
        bs = set(b)
        hits.append(len(bs.intersection(a)) / len(bs))
    return sum(hits) / len(hits)


def rel_error(o, o_ref):
    return ((o - o_ref).norm(dim=1) / o_ref.norm(dim=1)).mean().item()


def curve(workload="qwen_layer", n=None, budgets=(16, 32, 48, 68, 92, 136, 256, 512),
          modes=("sum", "per_head", "max"), layer=0, superblock=4096):
    w = synth.WORKLOADS[workload]
    if n is not None:
        w = synth.scaled(w, n=n)
    rows = w.kv_heads
    K = torch.stack([synth.keys(w, layer * rows + r, "cuda") for r in range(rows)])
    V = torch.stack([synth.values(w, layer * rows + r, "cuda") for r in range(rows)])
    q = synth.queries(w, layer, "cuda")
    k = min(w.k, w.n)
    index = F.pack(K, superblock)
    o_dense = dense_attention(q, K, V, w.group)
    out = {"workload": w.name, "n": w.n, "k": k, "kv_heads": rows, "group": w.group, "rows": []}
    for mode in modes:
        ref = exact_sets(q, K, w.group, k, mode)
        o_exact, _ = F.sparse_attn(q, K, V, ref, w.group, per_head=(mode == "per_head"))
        floor = rel_error(o_exact, o_dense)
        for B in budgets:
            st = F.DecodeStep(index, K, V, q, k, w.group, B, gqa=mode)
            idx, o, _ = st()
            # the same step with the keys of attention read back from the 4-bit index
            _, o4, _ = F.DecodeStep(index, None, V, q, k, w.group, B, gqa=mode, k_source="index")()
            out["rows"].append({"mode": mode, "budget": B, "recall": recall(idx, ref),
                                "error": rel_error(o, o_dense), "error_4bit_keys": rel_error(o4, o_dense),
                                "error_exact_k": floor, "error_vs_exact_k": rel_error(o, o_exact),
                                "error_4bit_keys_vs_exact_k": rel_error(o4, o_exact)})
    return out


def main():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--workload", default="qwen_layer")
    p.add_argument("--n", type=int, default=None)
    p.add_argument("--json", action="store_true", help="print the result as one JSON object")
    a = p.parse_args()
    res = curve(a.workload, a.n)
    if a.json:
        print(json.dumps(res))
        return
    print("workload %s: n=%d, k=%d, %d KV heads x %d query heads" % (res["workload"], res["n"], res["k"],
                                                                   res["kv_heads"], res["group"]))
    print("errors are ||o - o_ref|| / ||o_ref||, mean over query heads; o_ref = dense attention, or the")
    print("attention over the exact top-k keys of the same reading (columns 'vs exact-k')")
    print("%-9s %5s %7s %9s %9s %9s %12s %14s" % ("reading", "B", "recall", "error", "4b-K err", "exact-k",
                                                  "vs exact-k", "4b-K vs ex-k"))
    for r in res["rows"]:
        print("%-9s %5d %7.4f %9.4f %9.4f %9.4f %12.4f %14.4f" % (
            r["mode"], r["budget"], r["recall"], r["error"], r["error_4bit_keys"], r["error_exact_k"],
            r["error_vs_exact_k"], r["error_4bit_keys_vs_exact_k"]))


if __name__ == "__main__":
    main()
