"""The torch.autograd wrapper: its gradients are the library's backward on
the same inputs, bit for bit (deterministic mode), for one prompt group and
for several."""
import pytest
import torch

from shared_prompt_exact_dualkv_gb300 import synthetic

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("groups", [[(300, (200, 0, 131))], [(130, (70, 129)), (0, (50,)), (40, ())]])
def test_autograd_matches_direct_calls(groups):
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    Hq, Hkv, d = 4, 2, 128
    T = synthetic.group_rows(groups)
    x = synthetic.draw_inputs(T, Hq, Hkv, d, 3)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    if len(groups) == 1:
        out = D.dualkv_attention(qa, ka, va, P=groups[0][0], R_lens=groups[0][1], deterministic=True, num_splits=2)
    else:
        out = D.dualkv_attention(qa, ka, va, groups=groups, deterministic=True, num_splits=2)
    out.backward(do)
    ref_out, lse = D.forward_groups(q, k, v, groups)
    rdq, rdk, rdv = D.backward_groups(q, k, v, ref_out, do, lse, groups, deterministic=True, num_splits=2)
    assert torch.equal(out.detach(), ref_out)
    assert torch.equal(qa.grad, rdq) and torch.equal(ka.grad, rdk) and torch.equal(va.grad, rdv)


def test_calls_from_new_host_threads():
    """Library calls from threads whose first CUDA work they are (the
    autograd engine runs backward on such a worker thread).  The tensor-map
    encoder is a driver call that needs a current context, which the library
    binds itself.  Each thread's results equal the main thread's bit for bit
    (deterministic mode)."""
    import threading
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    P, R = 300, (200, 0, 131)
    x = synthetic.draw_inputs(P + sum(R), 4, 2, 128, 5)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    out, lse = D.forward(q, k, v, P, R)
    ref = D.backward(q, k, v, out, do, lse, P, R, deterministic=True)
    torch.cuda.synchronize()
    results, errors = [], []

    def work():
        try:
            o, l = D.forward(q, k, v, P, R)
            g = D.backward(q, k, v, o, do, l, P, R, deterministic=True)
            torch.cuda.synchronize()
            results.append((o, l) + tuple(g))
        except Exception as e:   # reported below, in the test's thread
            errors.append(e)

    threads = [threading.Thread(target=work) for _ in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for r in results:
        for a, b in zip(r, (out, lse) + tuple(ref)):
            assert torch.equal(a, b)


def test_autograd_after_other_library_work():
    """The autograd case again, after the library has run in the main thread
    (the order in which the worker thread first met a missing context)."""
    test_calls_from_new_host_threads()
    test_autograd_matches_direct_calls([(300, (200, 0, 131))])
