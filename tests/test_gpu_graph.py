"""The decode step (absorb -> decode -> out_proj) captured in a CUDA graph: the library's calls make
no host synchronisation, allocation or read-back when the caller passes every buffer, and the
device-built schedule (num_splits = -2) needs no host-side plan, so the whole step can be captured
once and replayed. Replays must equal eager calls bit for bit, also after new inputs are copied
into the captured buffers."""
import numpy as np
import pytest

import mla_inputs as mi

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("num_splits", [1, 3, -2])
def test_step_replays_in_a_cuda_graph(num_splits):
    import torch
    import mla_latent_kv_gb300 as mla
    B, Sq, H, lens = 4, 1, 32, [300, 64, 1000, 5]
    c = mi.e2e_case(B, Sq, H, lens, seed=40)
    dev = torch.device("cuda")
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa
    T = B * Sq
    qn = bf(c["q_nope"]).reshape(T, H, 128).contiguous()
    qp = bf(c["q_pe"]).reshape(T, H, 64).contiguous()
    wk, wv = bf(c["w_uk_t"]), bf(c["w_uv"])
    cache = torch.from_numpy(c["cache"]).to(dev)
    bt = torch.from_numpy(c["block_table"]).to(dev)
    sl = torch.from_numpy(np.asarray(c["seq_lens"], np.int32)).to(dev)
    max_len = max(lens)
    S = mla.resolve_num_splits(num_splits, B, Sq, H, max_len)
    ws = torch.empty(max(mla.workspace_bytes(B, Sq, H, S, mla.KV_BF16, max_len), 256), dtype=torch.uint8, device=dev)
    q = torch.empty((T, H, 576), dtype=torch.bfloat16, device=dev)
    ol = torch.empty((B, Sq, H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Sq, H), dtype=torch.float32, device=dev)
    o = torch.empty((T, H, 128), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        mla.absorb_q(qn, qp, wk, out=q)
        mla.decode(q.view(B, Sq, H, 576), cache, bt, sl, max_len, c["scale"], num_splits=num_splits, workspace=ws,
                   o_latent=ol, lse=lse, dev_status=status, num_blocks=c["num_blocks"])
        mla.out_proj(ol.view(T, H, 512), wv, out=o)

    step()
    torch.cuda.synchronize()
    o_eager, lse_eager = o.clone(), lse.clone()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        step()
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_eager) and torch.equal(lse, lse_eager)

    # new queries into the captured buffers: the replay follows them
    rng = np.random.default_rng(41)
    qn.copy_(bf(mi.normal_bf16(rng, (T, H, 128))).view(T, H, 128))
    g.replay()
    torch.cuda.synchronize()
    o_graph, lse_graph = o.clone(), lse.clone()
    step()
    torch.cuda.synchronize()
    assert torch.equal(o_graph, o) and torch.equal(lse_graph, lse)
    assert not torch.equal(o_graph, o_eager)
    assert int(status.item()) == 0
