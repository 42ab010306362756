"""The data-parallel split, on two `gloo` ranks on the CPU (no GPU).

Each rank takes its share of the work through the product's own host logic
(bit_nf4_quantized_38_b300.dp: token slices, group-aligned row shards, the
all-reduces) with the oracle doing the per-rank arithmetic, and the result is
compared with the single-rank oracle:
  * adapter gradients summed over token slices = the full batch's dA, dB
    (within the path's tolerance: the ranks' sums are added in fp32);
  * row-sharded quantization with the fp64 all-reduce of the absmax sum:
    packed codes, second-level codes, steps and the mean bit for bit."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    from bit_nf4_quantized_38_b300.workloads import normal_bf16, normal_with_outliers_bf16, bf16_bits
    M, N, K, r = 37, 96, 128, 8
    return dict(
        W=bf16_bits(normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, 5)),
        X=bf16_bits(normal_bf16((M, K), 1.0, 6)), A=bf16_bits(normal_bf16((K, r), 0.3, 7)),
        B=bf16_bits(normal_bf16((r, N), 0.01, 8)), dY=bf16_bits(normal_bf16((M, N), 1.0, 9)), s=2.0)


def _quant_weight():
    from bit_nf4_quantized_38_b300.workloads import bf16_bits, student_t4_bf16
    # 44 rows x 1152 cols = 18 blocks per row: shards must start on a 256-block group
    return bf16_bits(student_t4_bf16((44 * 3, 1152), 0.015, 11))


def _rank(rank, world, port, out):
    import torch
    import torch.distributed as dist
    for p in (ROOT, TESTS):
        sys.path.insert(0, p)
    from bit_nf4_quantized_38_b300 import dp
    from oracle import linear, nf4
    from oracle.bf16 import bf16_bits_to_f32
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        c = _case()
        m0, m1 = dp.token_slice(c["X"].shape[0], world, rank)
        dA, dB, _ = linear.lora_adapter_grads(c["dY"][m0:m1], c["X"][m0:m1], c["A"], c["B"], c["s"])
        tA = torch.from_numpy(dA.astype(np.float32))
        tB = torch.from_numpy(dB.astype(np.float32))
        dp.allreduce_adapter_grads_(tA, tB)

        W = _quant_weight()
        rows, cols = W.shape
        r0, r1 = dp.quant_row_shard(rows, cols, world, rank)
        w = bf16_bits_to_f32(W[r0:r1])
        am = nf4.block_absmax(w).reshape(-1)
        S, exact = nf4.exact_sum_f64(am)
        tS = torch.tensor([S], dtype=torch.float64)
        dp.allreduce_sum_(tS)
        total = rows * cols // 64
        mean = nf4.dq_mean_from_sum(float(tS[0]), total)
        code, step = nf4.double_quantize_codes(am, mean)
        packed = nf4.pack_nibbles(nf4.nf4_codes(w, am.reshape(r1 - r0, -1)))
        out.put((rank, (m0, m1), tA.numpy(), tB.numpy(), (r0, r1), packed, code, step, mean, exact))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_the_single_rank_oracle():
    sys.path.insert(0, TESTS)
    from parity import assert_close
    from oracle import linear, nf4
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted([q.get(timeout=120) for _ in procs], key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    c = _case()
    # token slices cover the batch once
    assert res[0][1] == (0, 18) and res[1][1] == (18, 37)
    dA, dB, _ = linear.lora_adapter_grads(c["dY"], c["X"], c["A"], c["B"], c["s"])
    for rank in range(2):
        assert_close(f"dp dA rank {rank}", res[rank][2], dA)
        assert_close(f"dp dB rank {rank}", res[rank][3], dB)
    assert np.array_equal(res[0][2], res[1][2]) and np.array_equal(res[0][3], res[1][3])
    # sharded quantization equals the unsharded oracle bit for bit
    W = _quant_weight()
    ref = nf4.quantize(W)
    (r0a, r1a), (r0b, r1b) = res[0][4], res[1][4]
    assert r0a == 0 and r1a == r0b and r1b == W.shape[0]
    assert (r1a * W.shape[1] // 64) % 256 == 0
    assert all(t[9] for t in res)
    assert np.array_equal(np.concatenate([res[0][5], res[1][5]]), ref["packed"])
    assert np.array_equal(np.concatenate([res[0][6], res[1][6]]), ref["code"])
    assert np.array_equal(np.concatenate([res[0][7], res[1][7]]).view(np.uint32), ref["step"].view(np.uint32))
    for rank in range(2):
        assert np.float32(res[rank][8]).view(np.uint32) == np.float32(ref["mean"]).view(np.uint32)


@pytest.mark.parametrize("rows,cols,world", [(132, 1152, 2), (4096, 4096, 8), (11008, 4096, 3), (7, 64, 4),
                                             (17920, 6656, 8)])
def test_row_shards_are_group_aligned_and_cover_the_weight(rows, cols, world):
    sys.path.insert(0, ROOT)
    from bit_nf4_quantized_38_b300 import dp
    shards = [dp.quant_row_shard(rows, cols, world, k) for k in range(world)]
    assert shards[0][0] == 0 and shards[-1][1] == rows
    for (a0, a1), (b0, b1) in zip(shards, shards[1:]):
        assert a1 == b0
    for r0, _ in shards:
        assert (r0 * cols // 64) % 256 == 0
    slices = [dp.token_slice(4096, world, k) for k in range(world)]
    assert slices[0][0] == 0 and slices[-1][1] == 4096
    assert max(b - a for a, b in slices) - min(b - a for a, b in slices) <= 1
