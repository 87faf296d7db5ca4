"""Parity at the workloads' full sizes, in the launch configuration the benchmark
times (one layer's 8 KV heads per decode step, the index and interleaved K/V in
host memory for the million-token workload), checked on
sampled rows that the oracle computes one by one:
pack, allocation and top-k bit-exact, scores and attention within tolerance."""
import numpy as np
import pytest
import torch

import oracle
from sparse_top_kv_fathom_gb300 import synth

pytestmark = pytest.mark.gpu

SCORE_RTOL = 1e-5
ATTN_ATOL = 2e-3


def _layer(F, w, layer, host, S):
    H = w.kv_heads
    rows = range(layer * H, (layer + 1) * H)
    K = torch.stack([synth.keys(w, r, "cuda") for r in rows])
    V = torch.stack([synth.values(w, r, "cuda") for r in rows])
    q = synth.queries(w, layer, "cuda")
    ix = F.pack(K, S)
    if host:  # as the benchmark lays it out: the index in pinned memory, K/V in fathom_host_alloc memory
        planes = ix.planes.cpu().pin_memory()
        meta = ix.meta.cpu().pin_memory()
        KV = F.host_empty((H, w.n, 2, 128), w.kv_dtype)
        KV.copy_(torch.stack([K, V], 2).cpu())
        sx = F.BitPlaneIndex(planes, meta, ix.var, ix.n, ix.rows, S)
        Ks, Vs, keep = KV[:, :, 0], KV[:, :, 1], (KV,)
    else:
        sx, Ks, Vs, keep = ix, K, V, ()
    return K, V, q, ix, sx, Ks, Vs, keep


@pytest.mark.parametrize("name,layer,sample,host,S", [
    ("million", 0, (0,), True, 4096),
    ("million", 35, (7,), True, 4096),
    ("decode36", 17, (2,), False, 4096),
    ("sessions", 11, (1, 6), False, 4096),
    ("qwen_layer", 0, (0, 4), False, 1024),
])
def test_full_size_sampled_rows(gpu_lib, name, layer, sample, host, S):
    F = gpu_lib
    w = synth.WORKLOADS[name]
    budgets = synth.row_budgets(w)[layer * w.kv_heads:(layer + 1) * w.kv_heads]
    budget = torch.tensor(budgets.numpy().astype(np.int16)).cuda() if w.per_row_budget else int(budgets[0])
    K, V, q, ix, sx, Ks, Vs, keep = _layer(F, w, layer, host, S)
    step = F.DecodeStep(sx, Ks, Vs, q, w.k, w.group, budget)
    idx, out, outb = step()
    bits, qbar = F.allocate(q, ix.var, budget, w.group)
    scores = F.scan(sx, bits, qbar)
    torch.cuda.synchronize()
    G = w.group
    for r in sample:
        Kr = K[r:r + 1].float().cpu().numpy()
        planes, meta, var = oracle.pack(Kr, S)
        assert np.array_equal(ix.planes[r:r + 1].cpu().numpy().view(np.uint32), planes), "planes"
        assert np.array_equal(ix.meta[r:r + 1].cpu().numpy().view(np.uint16), meta), "meta"
        assert np.array_equal(ix.var[r:r + 1].cpu().numpy(), var), "var"
        qr = q[r * G:(r + 1) * G].float().cpu().numpy()
        b_r = int(budgets[r])
        obits, oqbar = oracle.allocate(qr, var, b_r, G)
        assert np.array_equal(bits[r:r + 1].cpu().numpy(), obits), "allocation"
        ref, l1 = oracle.scan(planes, meta, obits, oqbar, w.n, S)
        s_r = scores[r:r + 1].cpu().numpy()
        assert (np.abs(s_r.astype(np.float64) - ref) <= SCORE_RTOL * l1).all(), "scores"
        oi = oracle.topk_f32(s_r, w.k)
        assert np.array_equal(idx[r:r + 1].cpu().numpy(), oi), "top-k"
        oo = oracle.sparse_attn(qr, Kr, V[r:r + 1].float().cpu().numpy(), oi, G)
        got = out[r * G:(r + 1) * G].cpu().numpy()
        assert np.abs(got - oo).max() <= ATTN_ATOL, "attention"
        rne = torch.from_numpy(got).to(torch.bfloat16).float().numpy()
        assert (np.abs(outb[r * G:(r + 1) * G].float().cpu().numpy() - rne) <= np.abs(rne) * 2.0 ** -7 + 1e-38).all()
    for t in keep:
        F.host_release(t)
