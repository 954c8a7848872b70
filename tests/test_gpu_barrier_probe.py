"""The grid-barrier probe (ck_probe_grid_barrier): every scheme crosses its
barriers with no wait running out, at the recurrence kernels' shape (two
256-thread CTAs per SM); bad arguments are refused before any launch."""
import pytest
import torch

pytestmark = pytest.mark.gpu

SCHEMES = [("BARRIER_COUNTER", 1), ("BARRIER_COUNTER_RETURNING", 1), ("BARRIER_COUNTER_RELAXED", 1),
           ("BARRIER_FLAG", 1), ("BARRIER_FLAGS8", 1), ("BARRIER_CLUSTER_SYNC", 2),
           ("BARRIER_CLUSTER_SYNC", 8), ("BARRIER_CLUSTER_MBARRIER", 2), ("BARRIER_CLUSTER_MBARRIER", 4),
           ("BARRIER_CLUSTER_MBARRIER", 8)]


def _buffers(ctas, rows_per_cta):
    from sparse_graph_recurrent_gb300 import _ck
    dev = torch.device("cuda")
    rows = torch.zeros(max(ctas * rows_per_cta * 32, 1), dtype=torch.float32, device=dev)
    words = torch.zeros(_ck.PROBE_BARRIER_WORDS, dtype=torch.int32, device=dev)
    status = torch.full((1,), 7, dtype=torch.int32, device=dev)
    return rows, words, status


@pytest.mark.parametrize("name,cluster", SCHEMES, ids=[f"{n.lower()}_{c}" for n, c in SCHEMES])
def test_scheme_crosses_every_barrier(name, cluster):
    from sparse_graph_recurrent_gb300 import _ck
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ctas, crossings, rpc = 2 * sms, 300, 16
    rows, words, status = _buffers(ctas, rpc)
    _ck.ck_probe_grid_barrier(getattr(_ck, name), ctas, cluster, crossings, rpc, rows, words, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0  # cleared by the call, untouched by a crossing that completed
    # every CTA wrote its rows on the last crossing: value (crossings - 1 + i) at position i
    last = rows[: ctas * rpc * 32].view(ctas, rpc * 32).cpu()
    expect = torch.arange(rpc * 32, dtype=torch.float32) + (crossings - 1)
    assert torch.equal(last, expect.expand(ctas, -1))
    if name in ("BARRIER_COUNTER", "BARRIER_COUNTER_RELAXED"):
        assert int(words[0].item()) == ctas * crossings  # one arrival per CTA per crossing
    elif name in ("BARRIER_CLUSTER_SYNC", "BARRIER_CLUSTER_MBARRIER"):
        assert int(words[0].item()) == ctas // cluster * crossings


def test_single_cta_and_no_rows():
    from sparse_graph_recurrent_gb300 import _ck
    _, words, status = _buffers(1, 0)
    _ck.ck_probe_grid_barrier(_ck.BARRIER_COUNTER, 1, 1, 50, 0, None, words, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and int(words[0].item()) == 50


@pytest.mark.parametrize("scheme,ctas,cluster,crossings,rpc", [
    (7, 8, 1, 10, 0),        # unknown scheme
    (-1, 8, 1, 10, 0),
    (0, 8, 2, 10, 0),        # cluster only for the cluster schemes
    (5, 8, 1, 10, 0),        # the cluster schemes need 2, 4 or 8
    (5, 9, 2, 10, 0),        # ctas a multiple of the cluster
    (0, 0, 1, 10, 0),
    (0, 8, 1, 0, 0),
    (0, 8, 1, 10, 65),       # at most 64 rows per CTA
])
def test_bad_arguments_are_refused(scheme, ctas, cluster, crossings, rpc):
    from sparse_graph_recurrent_gb300 import _ck
    rows, words, status = _buffers(16, 65)  # large enough that the binding passes it on
    with pytest.raises(_ck.CKError) as ei:
        _ck.ck_probe_grid_barrier(scheme, ctas, cluster, crossings, rpc, rows, words, status)
    assert ei.value.name == "CK_ERR_INVALID_ARG"


def test_more_ctas_than_fit_are_refused():
    from sparse_graph_recurrent_gb300 import _ck
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows, words, status = _buffers(1, 0)
    with pytest.raises(_ck.CKError) as ei:
        _ck.ck_probe_grid_barrier(_ck.BARRIER_COUNTER, 16 * sms, 1, 10, 0, None, words, status)
    assert ei.value.name == "CK_ERR_UNSUPPORTED"
