"""The form dispatcher against live measurements: on one causal prompt at
H = 32 (DeepSeek-V3.2 at TP4) the form it picks must be within 15 % of the
fastest measured form, at a length where masked MHA wins and at one where the
grouped form wins."""
import pytest

from gpu_util import need_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.mark.parametrize("L", [8192, 32768])
def test_dispatch_pick_is_fastest(L):
    import bench
    import dsa_sparse_mla_prefill_gb300 as dsa
    dev = torch.device("cuda", 0)
    flush_buf = torch.empty(bench.FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    res = bench.measure_forms(L, dev, torch.cuda.current_stream(dev), lambda: flush_buf.zero_(), 5, 3)
    assert res["device_errors"][1] == 0 and res["device_errors"][2] == 0
    measured = {"per_token": res["per_token_ms"], "grouped": res["union_ms"] + res["grouped_ms"],
                "masked": res["key_mask_ms"] + res["masked_ms"]}
    form, pred, _ = dsa.dsa_choose_form([L], [L], 32, 2048, 576, (192, 128), union_rows=res["union_rows"])
    assert measured[form] <= 1.15 * min(measured.values()), (form, measured, pred)
    for f in dsa.FORMS:   # the model's times themselves within 25 % of the measurement
        assert pred[f] == pytest.approx(measured[f], rel=0.25), (f, pred, measured)
