"""Data-parallel split of the QLoRA linear over ranks (one process per GPU).

The QLoRA project page trains on several GPUs through Accelerate; in data
parallel every rank holds the same frozen NF4 weight and the same adapter A,
B, and processes its own tokens.  The only exchange the layer needs is:

  * training: the adapter gradients dA = s X^T (dY B^T) and dB = s (X A)^T dY
    are sums over tokens, so each rank's gradients on its tokens are summed
    over ranks (one all-reduce of r (K + N) floats per linear); Y and dX stay
    on the rank that owns the tokens;
  * quantization: rows are independent; the double-quant mean needs the sum
    of all block absmax values (an fp64 all-reduce of one number, exact for
    real weights) and the total block count.

Host logic only: the arithmetic runs in the CUDA library (qlora.py) and the
sums in torch.distributed (NCCL on GPUs, gloo on CPU tensors).
"""
import math

import torch
import torch.distributed as dist

DQ_GROUP_BLOCKS = 256
BLOCK = 64


def token_slice(M, world, rank):
    """Rows [m0, m1) of an M-token batch that `rank` of `world` processes
    when one global batch is split (contiguous, sizes differ by at most 1)."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    return (M * rank) // world, (M * (rank + 1)) // world


def quant_row_step(cols):
    """Rows per shard must be a multiple of this so that every shard starts on
    a 256-block double-quant group boundary of the whole tensor."""
    if cols % BLOCK:
        raise ValueError(f"cols {cols} not a multiple of {BLOCK}")
    bpr = cols // BLOCK
    return DQ_GROUP_BLOCKS // math.gcd(bpr, DQ_GROUP_BLOCKS)


def quant_row_shard(rows, cols, world, rank):
    """Rows [r0, r1) of a weight that `rank` quantizes: group-aligned starts,
    as even as the alignment allows (the last shard takes the remainder)."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    step = quant_row_step(cols)
    units = -(-rows // step)
    u0, u1 = (units * rank) // world, (units * (rank + 1)) // world
    return min(rows, u0 * step), min(rows, u1 * step)


def allreduce_sum_(t, group=None):
    """In-place sum over the ranks (no-op when torch.distributed is not up)."""
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return t


def allreduce_adapter_grads_(dA, dB, group=None):
    """dA, dB of this rank's tokens -> the sums over all ranks' tokens."""
    allreduce_sum_(dA, group)
    allreduce_sum_(dB, group)
    return dA, dB


def dp_nf4_quantize(ql, W_shard, total_blocks, dq_blocksize=256, group=None, stream=None):
    """Quantize this rank's rows of a weight; the double-quant mean comes from
    the absmax sum over all ranks' rows (see nf4_quantize_shard_begin/end)."""
    q, ws, partial = ql.nf4_quantize_shard_begin(W_shard, dq_blocksize=dq_blocksize, stream=stream)
    if dq_blocksize:
        allreduce_sum_(partial, group)
    return ql.nf4_quantize_shard_end(q, ws, total_blocks, stream=stream)


def dp_linear_bwd(ql, dY, X, XA, q, A, B, scale, group=None, **kw):
    """Backward on this rank's tokens, then the adapter gradients summed over
    ranks; dX stays local.  Returns (dX, dA, dB)."""
    dX, dA, dB = ql.qlora_linear_bwd(dY, X, XA, q, A, B, scale, **kw)
    allreduce_adapter_grads_(dA, dB, group)
    return dX, dA, dB
