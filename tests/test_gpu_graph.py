"""The entry points copy nothing host-to-device and pass their schedule and
tensor maps by value, so a forward + backward can be captured in a CUDA graph
and replayed on new inputs written into the same buffers.  The replay must
give the bits of eager calls on those inputs (deterministic reduction mode;
the many-tile case is split into several launches per kernel)."""
import pytest
import torch

from shared_prompt_exact_dualkv_gb300 import synthetic

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("groups,Hq,Hkv,d", [([(300, (200, 0, 131))], 4, 2, 128),
                                             ([(16384, (4096,) * 16)] * 8, 2, 1, 64)])
def test_graph_replay_matches_eager(groups, Hq, Hkv, d):
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    T = synthetic.group_rows(groups)
    scale = d ** -0.5
    bufs = [t.cuda() for t in (lambda x: (x.q, x.k, x.v, x.dout))(synthetic.draw_inputs(T, Hq, Hkv, d, 1))]
    q, k, v, do = bufs
    out = torch.empty_like(q)
    lse = torch.empty((Hq, T), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(D.dualkv_bwd_groups_workspace_bytes(groups, Hq, Hkv, d, True, 2), dtype=torch.uint8,
                     device="cuda")

    def step():
        D.dualkv_fwd_groups(q, k, v, groups, out, lse, scale)
        D.dualkv_bwd_groups(q, k, v, out, do, lse, groups, scale, True, ws, dq, dk, dv, num_splits=2)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    # new inputs into the captured buffers, then replay
    new = synthetic.draw_inputs(T, Hq, Hkv, d, 2)
    for dst, src in zip(bufs, (new.q, new.k, new.v, new.dout)):
        dst.copy_(src)
    g.replay()
    torch.cuda.synchronize()
    assert D.dualkv_last_device_error() == (D.DUALKV_OK, 0)
    replayed = [t.clone() for t in (out, lse, dq, dk, dv)]
    step()
    torch.cuda.synchronize()
    for a, b in zip(replayed, (out, lse, dq, dk, dv)):
        assert torch.equal(a, b)
