"""Parameter layouts of the models the ZeRO pages size their examples on.

Each workload is a list of tensor element counts in declaration order (what
gets flattened), a ZeRO-3 unit id per tensor (one unit per transformer block,
unit 0 = the root unit holding embeddings, final norm and head, as in
"別再複製本可分片的東西：ZeRO 與 FSDP", "FSDP：同樣的想法，以層為單位"), and the
step settings the benchmark and parity tests use.

Models:
  * GPT-2 1.5B (the example of "ZeRO: Memory Optimizations Toward Training
    Trillion Parameter Models" reading notes §2.1: 3 + 3 + 18 = 24 GB of model
    states): 48 blocks, d = 1600, ffn 6400, vocab 50257, context 1024, tied head;
  * GPT-2 small (124M), GPT-2 medium (350M, plus one 1-element tensor so that
    Psi is odd), Llama-style 7B (the 7B of "第 5 课：ZeRO 与 FSDP", its numeric
    example: 32 blocks, d = 4096, SwiGLU ffn 11008, vocab 32000, untied head);
  * a tiny four-tensor buffer for fast parity runs.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

BF16 = 0
FP16 = 1


def gpt2_tensors(n_layer: int, d: int, ffn: int, vocab: int = 50257, ctx: int = 1024):
    """GPT-2 with a tied LM head: wte, wpe, blocks, ln_f."""
    numels: List[int] = [vocab * d, ctx * d]
    units: List[int] = [0, 0]
    for l in range(n_layer):
        block = [d, d,                 # ln_1 weight, bias
                 d * 3 * d, 3 * d,     # attn c_attn weight, bias
                 d * d, d,             # attn c_proj weight, bias
                 d, d,                 # ln_2 weight, bias
                 d * ffn, ffn,         # mlp c_fc weight, bias
                 ffn * d, d]           # mlp c_proj weight, bias
        numels += block
        units += [l + 1] * len(block)
    numels += [d, d]                   # ln_f weight, bias
    units += [0, 0]
    return numels, units


def llama_tensors(n_layer: int = 32, d: int = 4096, ffn: int = 11008, vocab: int = 32000):
    """Llama-style decoder with RMSNorm, SwiGLU MLP and an untied head."""
    numels: List[int] = [vocab * d]
    units: List[int] = [0]
    for l in range(n_layer):
        block = [d,                        # attention RMSNorm
                 d * d, d * d, d * d, d * d,   # wq, wk, wv, wo
                 d,                        # MLP RMSNorm
                 d * ffn, d * ffn, ffn * d]    # w_gate, w_up, w_down
        numels += block
        units += [l + 1] * len(block)
    numels += [d, vocab * d]               # final norm, untied head
    units += [0, 0]
    return numels, units


@dataclass
class Workload:
    name: str
    numels: List[int]
    unit_of_tensor: List[int]
    n_d: int
    stage: int
    dtype: int                      # BF16 or FP16 gradients / parameters
    bucket_elems: int               # <= 0: one bucket
    grad_std: float
    per_tensor_scale: bool          # multiply each tensor's grads by U(0.1, 10)
    master_std: float = 0.02
    max_norm: float = 0.0           # <= 0: no clipping
    loss_scale: float = 1.0
    dynamic_scale: bool = False
    growth_interval: int = 2000
    steps: int = 3
    inf_step: Optional[int] = None  # 1-based step whose rank-3 replica gets +inf
    inf_rank: int = 3
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    extra: dict = field(default_factory=dict)

    @property
    def psi(self) -> int:
        return sum(self.numels)

    def fused(self) -> bool:
        """No clipping and no loss scaler: reduce, update and gather in one pass."""
        return self.max_norm <= 0 and not self.dynamic_scale and self.loss_scale == 1.0


def tiny() -> Workload:
    numels = [1000 * 512, 512, 487 * 1000, 2491]
    return Workload("tiny: Psi=1,002,003 (4 tensors), N_d=4, ZeRO-2, bf16",
                    numels, [0, 0, 1, 1], n_d=4, stage=2, dtype=BF16, bucket_elems=0,
                    grad_std=1e-3, per_tensor_scale=False, steps=3)


def gpt2_small() -> Workload:
    numels, units = gpt2_tensors(12, 768, 3072)
    return Workload("GPT-2 small 124M, N_d=8, ZeRO-1, bf16, bucket 5e6",
                    numels, units, n_d=8, stage=1, dtype=BF16, bucket_elems=5_000_000,
                    grad_std=1e-3, per_tensor_scale=True, steps=10)


def gpt2_xl() -> Workload:
    numels, units = gpt2_tensors(48, 1600, 6400)
    return Workload("GPT-2 1.5B, N_d=8, ZeRO-2, fp16 grads, loss scale 2^16 dynamic, clip 1.0, bucket 5e8",
                    numels, units, n_d=8, stage=2, dtype=FP16, bucket_elems=500_000_000,
                    grad_std=1e-3, per_tensor_scale=True, max_norm=1.0,
                    loss_scale=65536.0, dynamic_scale=True, steps=10, inf_step=4, inf_rank=3)


def gpt2_xl_block() -> Workload:
    """One GPT-2 1.5B transformer block (30.7M parameters) with the 1.5B
    run's settings: the same kernels on a buffer small enough (~1.5 GB on the
    device, still far above L2) for multi-pass profiler captures."""
    numels, units = gpt2_tensors(1, 1600, 6400)
    numels, units = numels[2:-2], [0] * (len(numels) - 4)
    return Workload("one GPT-2 1.5B block (30.7M), N_d=8, ZeRO-2, fp16, loss scale 2^16, clip 1.0",
                    numels, units, n_d=8, stage=2, dtype=FP16, bucket_elems=500_000_000,
                    grad_std=1e-3, per_tensor_scale=True, max_norm=1.0,
                    loss_scale=65536.0, dynamic_scale=True, steps=10)


def llama7b() -> Workload:
    numels, units = llama_tensors()
    return Workload("Llama-style 7B, N_d=2, ZeRO-3 (33 units), bf16",
                    numels, units, n_d=2, stage=3, dtype=BF16, bucket_elems=0,
                    grad_std=5e-4, per_tensor_scale=False, steps=10)


def llama7b_block() -> Workload:
    """One Llama-style 7B block (202M parameters) as ZeRO-3 unit 1 behind a
    4096-element root unit (the final norm), with the 7B run's settings: the
    same per-unit gather and fused kernels on ~4 GB of device memory, small
    enough for multi-pass profiler captures and still far above L2."""
    numels, units = llama_tensors(n_layer=1)
    block = numels[1:-2]
    return Workload("one Llama-style 7B block (202M) + final norm, N_d=2, ZeRO-3 (2 units), bf16",
                    [4096] + block, [0] + [1] * len(block), n_d=2, stage=3, dtype=BF16,
                    bucket_elems=0, grad_std=5e-4, per_tensor_scale=False, steps=10)


def gpt2_medium_odd(n_d: int = 8, stage: int = 2, bucket_elems: int = 5_000_000) -> Workload:
    numels, units = gpt2_tensors(24, 1024, 4096)
    numels = numels + [1]
    units = units + [0]
    return Workload("GPT-2 medium 350M + 1 (odd Psi), N_d=%d, ZeRO-%d, bf16, bucket %d"
                    % (n_d, stage, bucket_elems),
                    numels, units, n_d=n_d, stage=stage, dtype=BF16, bucket_elems=bucket_elems,
                    grad_std=1e-3, per_tensor_scale=True, steps=3)


ALL = {"tiny": tiny, "gpt2_small": gpt2_small, "gpt2_xl": gpt2_xl, "llama7b": llama7b,
       "gpt2_xl_block": gpt2_xl_block, "llama7b_block": llama7b_block,
       "gpt2_medium": gpt2_medium_odd}
