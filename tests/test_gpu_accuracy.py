"""The synthetic accuracy curve (attention error and recall of the exact top-k against the
budget, for the three GQA readings): sanity properties that hold on any data."""
import pytest

pytestmark = pytest.mark.gpu


def test_accuracy_curve_properties(gpu_lib):
    from sparse_top_kv_fathom_gb300 import accuracy
    res = accuracy.curve("qwen_layer", n=8192, budgets=(16, 92, 512))
    by = {(r["mode"], r["budget"]): r for r in res["rows"]}
    for mode in ("sum", "per_head", "max"):
        lo, mid, hi = by[(mode, 16)], by[(mode, 92)], by[(mode, 512)]
        for r in (lo, mid, hi):
            assert 0.0 <= r["recall"] <= 1.0
            assert r["error"] >= 0.0
            # no k-key selection beats the exact top-k of the true logits by much
            assert r["error"] >= r["error_exact_k"] * 0.9
        # more bits per key never hurt much and help overall
        assert hi["recall"] >= lo["recall"]
        assert hi["recall"] > 0.5
        assert hi["error"] <= lo["error"] * 1.05
