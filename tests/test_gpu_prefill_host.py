"""GPU check of the host-buffer prefill (swiattn_prefill_host): from pinned
or pageable host tensors it must return exactly what swiattn_prefill returns
on the same inputs in device memory (outputs and lse bit for bit), for bf16
with and without anchors and for fp32."""
import pytest
import torch

import swiattn_inputs as inp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    import sliding_window_attention_router_gb300 as m
    return m


@pytest.mark.parametrize("B,N,Hq,Hkv,W,S,pinned", [
    (1, 4096, 16, 16, 1024, 0, True),
    (2, 777, 8, 2, 100, 64, True),
    (1, 300, 4, 4, 64, 0, False),
])
def test_host_equals_device_bf16(swa, B, N, Hq, Hkv, W, S, pinned):
    g = inp._gen(N + W)
    q, k, v = inp.attention_qkv(B, N, Hq, Hkv, 128, torch.bfloat16, g)
    gate = torch.stack([inp.run_gates(N, 0.2, g) for _ in range(B)])
    if pinned:
        q, k, v, gate = (t.pin_memory() for t in (q, k, v, gate))
    o_h, lse_h = swa.prefill_host(q, k, v, gate, W, n_anchor=S, want_lse=True)
    torch.cuda.synchronize()
    o_d, lse_d = swa.prefill(q.cuda(), k.cuda(), v.cuda(), gate.cuda(), W, n_anchor=S,
                             want_lse=True)
    torch.cuda.synchronize()
    assert swa.get_device_error() == 0
    assert torch.equal(o_h.view(torch.int16), o_d.cpu().view(torch.int16))
    assert torch.equal(lse_h, lse_d.cpu())


def test_host_equals_device_fp32(swa):
    g = inp._gen(5)
    q, k, v = inp.attention_qkv(1, 256, 2, 2, 64, torch.float32, g)
    gate = inp.bernoulli_gates((1, 256), 0.13, g)
    o_h = swa.prefill_host(q, k, v, gate, 32)
    torch.cuda.synchronize()
    o_d = swa.prefill(q.cuda(), k.cuda(), v.cuda(), gate.cuda(), 32)
    assert torch.equal(o_h, o_d.cpu())


def test_calls_alternating_two_streams(swa):
    """The bench's end-to-end figure issues host-buffer calls back to back on
    two streams, each with its own workspace and output, so two calls (their
    copies and their kernels) can run at once.  Each result must equal the
    same call made alone, bit for bit."""
    dev = torch.device("cuda", 0)
    B, N, H, W = 1, 4096, 8, 512
    cases = []
    for seed in (11, 12, 13, 14):
        g = inp._gen(seed)
        q, k, v = inp.attention_qkv(B, N, H, H, 128, torch.bfloat16, g)
        gate = inp.run_gates(N, 0.13, g).reshape(B, N)
        cases.append(tuple(t.pin_memory() for t in (q, k, v, gate)))
    alone = []
    for q, k, v, gate in cases:
        o = swa.prefill_host(q, k, v, gate, W)
        torch.cuda.synchronize()   # the host output is valid once the stream has passed the call
        alone.append(o.clone())
    ws_bytes = swa.prefill_host_workspace(B, N, H, H, 128, W, torch.bfloat16)
    lanes = [(torch.cuda.Stream(dev), torch.empty(ws_bytes, dtype=torch.uint8, device=dev))
             for _ in range(2)]
    outs = [torch.empty(cases[0][0].shape, dtype=torch.bfloat16, pin_memory=True) for _ in cases]
    main = torch.cuda.current_stream(dev)
    for st, _ in lanes:
        st.wait_stream(main)
    for rep in range(3):
        for i, (q, k, v, gate) in enumerate(cases):
            st, ws = lanes[i % 2]
            with torch.cuda.stream(st):
                swa.prefill_host(q, k, v, gate, W, out=outs[i], workspace=ws, device=dev)
        for st, _ in lanes:
            main.wait_stream(st)
        torch.cuda.synchronize()
        assert swa.get_device_error() == 0
        for i in range(len(cases)):
            assert torch.equal(outs[i].view(torch.int16), alone[i].view(torch.int16)), (rep, i)
