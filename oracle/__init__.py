"""CPU oracle for the QLoRA NF4 linear hot path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously-correct
restatement of what the method computes, in fp64 (numpy) wherever the method
does floating point, used to check the CUDA library.  Only the test suite, the
smoke check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import it.  It shares no code, table or constant with the CUDA path, and the
product path never calls it.

Sources (titles of the pages the method is described on):
  * "QLoRA: Efficient Finetuning of Quantized LLMs" (arXiv 2305.14314 abstract
    page): 4-bit NormalFloat, double quantization, backprop through a frozen
    4-bit model into LoRA adapters.
  * The Chinese news write-up of QLoRA/Guanaco: NF4 is information-theoretically
    optimal for normally distributed weights; double quantization quantizes the
    quantization constants, saving about 0.37 bit per parameter (about 3 GB at
    65B); adapters on every layer.
  * The LoRA tutorial (Lit-LLaMA, Chinese translation): h = W x + dW x with
    dW = W_A W_B, W_A of size A x r and W_B of size r x B, a scale alpha on the
    low-rank branch, W_B initialised to zero, and the merge W' = W + W_A W_B.

Modules:
  nf4     -- codebook, blockwise absmax, NF4 code + nibble pack, double
             quantization of the absmax constants, dequantization.
  linear  -- forward and backward of the frozen-NF4 linear with a LoRA adapter.
  fp8     -- the same forward with the main product on E4M3 operands.
  bf16    -- IEEE round-to-nearest-even to bfloat16 and back.

Parity status of each function is stated in its docstring; the readings taken
where the pages are silent are listed in the module docstrings.
"""
