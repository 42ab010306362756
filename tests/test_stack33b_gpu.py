"""The LLaMA-33B stack at full size: 60 layers x 7 linears (6656 x 6656,
17920 x 6656, 6656 x 17920), r = 64, M = 2048 tokens, 16.6 GB of NF4 weights
resident at once.  The forward runs through all 420 linears in order, then
the backward in reverse, back to back with one workspace; three linears
spread over the stack are checked against the fp64 oracle (Y and dX on 32
sampled token rows, XA, dA and dB in full).  Weights and inputs are drawn on
the device from seeded generators; the checked ones are copied to the host
for the oracle."""
import numpy as np
import pytest
import torch

from oracle import linear, nf4
from parity import assert_close

pytestmark = pytest.mark.gpu

CHECKED = (0, 29 * 7 + 5, 59 * 7 + 6)  # layer 0 q_proj, layer 29 up_proj, layer 59 down_proj


@pytest.fixture(scope="module")
def ql():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_38_b300 import qlora
    return qlora


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def test_llama33b_stack_full_size(ql):
    from bit_nf4_quantized_38_b300.workloads import bf16_bits, case_inputs, case_weight, llama33b_stack
    dev = torch.device("cuda")
    cases = llama33b_stack().cases
    assert len(cases) == 420
    qs, w_bits = [], {}
    for i, c in enumerate(cases):
        W = case_weight(c, device=dev)
        qs.append(ql.nf4_quantize(W))
        if i in CHECKED:
            w_bits[i] = bf16_bits(W)
        del W
    torch.cuda.synchronize()
    ql.device_status()
    assert sum(q.nbytes() for q in qs) > 16e9

    M, r = cases[0].M, cases[0].r
    N_max = max(c.N for c in cases)
    K_max = max(c.K for c in cases)
    ws = torch.empty(max(ql.workspace_size(ql.OP_LINEAR_FWD, M, N_max, K_max, r),
                         ql.workspace_size(ql.OP_LINEAR_BWD, M, N_max, K_max, r)), dtype=torch.uint8, device=dev)
    xas, got = [], {}
    for i, c in enumerate(cases):  # forward, in order
        X, A, B, _ = case_inputs(c, device=dev)
        Y, XA = ql.qlora_linear_fwd(X, qs[i], A, B, c.scale, ws=ws)
        xas.append(XA)
        if i in CHECKED:
            got[i] = {"Y": Y.cpu(), "XA": XA.cpu()}
    for i in reversed(range(len(cases))):  # backward, in reverse
        c = cases[i]
        X, A, B, dY = case_inputs(c, device=dev)
        dX, dA, dB = ql.qlora_linear_bwd(dY, X, xas[i], qs[i], A, B, c.scale, ws=ws)
        if i in CHECKED:
            got[i].update(dX=dX.cpu(), dA=dA.cpu(), dB=dB.cpu(),
                          inputs=[bf16_bits(t) for t in (X, A, B, dY)])
    torch.cuda.synchronize()
    ql.device_status()
    del qs, xas, ws
    torch.cuda.empty_cache()

    for i in CHECKED:
        c, g = cases[i], got[i]
        Xb, Ab, Bb, dYb = g["inputs"]
        Wh = nf4.dequantize(nf4.quantize(w_bits[i], 64, 256))
        rows = np.sort(np.random.default_rng(i).choice(c.M, 32, replace=False))
        Yr, _ = linear.lora_forward(Xb[rows], Wh, Ab, Bb, c.scale)
        assert_close(f"{c.name} Y rows", f64(g["Y"])[rows], Yr)
        dXr, _, _, _ = linear.lora_backward(dYb[rows], Xb[rows], Wh, Ab, Bb, c.scale)
        assert_close(f"{c.name} dX rows", f64(g["dX"])[rows], dXr)
        del Wh
        dAr, dBr, XAr = linear.lora_adapter_grads(dYb, Xb, Ab, Bb, c.scale)
        assert_close(f"{c.name} XA", f64(g["XA"]), XAr)
        assert_close(f"{c.name} dA", f64(g["dA"]), dAr)
        assert_close(f"{c.name} dB", f64(g["dB"]), dBr)
