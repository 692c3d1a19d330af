"""Named synthetic workloads of the decode MoE expert block (shapes only, no arithmetic).

Each workload is a layer shape plus a layer count and a token count.  The shapes follow the MoE
models the pages measure: the qwen3-30b-a3b MoE (2048 hidden, 768 expert width, 128 experts,
top-8), the qwen1.5-moe-a2.7b MoE (60 experts, top-4, one wide shared expert behind a sigmoid
gate), a 512-expert top-10 model with a narrow gated shared expert, and a dots.llm1-like model
(4096 hidden, 6-bit down projection, two ungated shared experts).
"""
from __future__ import annotations

import dataclasses


@dataclasses.dataclass(frozen=True)
class Shape:
    name: str
    din: int
    dff: int
    n_experts: int
    top_k: int
    bits_gate: int
    bits_up: int
    bits_down: int
    n_shared: int = 0
    dff_shared: int = 0
    bits_shared: int = 4
    shared_gate: int = 0       # 0: shared scalar 1; 1: sigmoid(x . g)
    layers: int = 1
    tokens: int = 1
    seed: int = 0x5EED0001

    def proj_bytes(self, rows: int, cols: int, bits: int) -> int:
        """Packed bytes of one projection: codes + fp16 scale and bias per 64 codes."""
        return rows * cols * bits // 8 + (rows * cols // 64) * 4

    def expert_bytes(self) -> int:
        return (self.proj_bytes(self.dff, self.din, self.bits_gate)
                + self.proj_bytes(self.dff, self.din, self.bits_up)
                + self.proj_bytes(self.din, self.dff, self.bits_down))

    def shared_bytes(self) -> int:
        if not self.n_shared:
            return 0
        one = (2 * self.proj_bytes(self.dff_shared, self.din, self.bits_shared)
               + self.proj_bytes(self.din, self.dff_shared, self.bits_shared))
        return self.n_shared * one

    def layer_weight_bytes(self) -> int:
        return self.n_experts * self.expert_bytes() + self.shared_bytes()

    def with_(self, **kw) -> "Shape":
        return dataclasses.replace(self, **kw)


# Single MoE layer, qwen3-30b-a3b shape, 4-bit, no shared expert.
QWEN3_30B_A3B_4BIT_LAYER = Shape("qwen3-30b-a3b moe layer, 4-bit", din=2048, dff=768,
                                 n_experts=128, top_k=8, bits_gate=4, bits_up=4, bits_down=4,
                                 seed=0x5EED0001)

# Single layer, qwen1.5-moe-a2.7b shape: 60 experts, top-4, one 5632-wide shared expert
# scaled by sigmoid(x . g).
QWEN15_MOE_A27B_LAYER = Shape("qwen1.5-moe-a2.7b layer, 4-bit, gated shared expert", din=2048,
                              dff=1408, n_experts=60, top_k=4, bits_gate=4, bits_up=4,
                              bits_down=4, n_shared=1, dff_shared=5632, bits_shared=4,
                              shared_gate=1, seed=0x5EED0002)

# 48-layer stack, qwen3-30b-a3b shape, 8-bit codes (about 29 GB of codes).
QWEN3_30B_A3B_8BIT_STACK = Shape("qwen3-30b-a3b moe stack, 48 layers, 8-bit", din=2048, dff=768,
                                 n_experts=128, top_k=8, bits_gate=8, bits_up=8, bits_down=8,
                                 layers=48, seed=0x5EED0003)

# 40-layer stack: 512 experts, top-10, one narrow gated shared expert.
E512_TOP10_STACK = Shape("512-expert top-10 stack, 40 layers, 4-bit, gated shared expert",
                         din=2048, dff=512, n_experts=512, top_k=10, bits_gate=4, bits_up=4,
                         bits_down=4, n_shared=1, dff_shared=512, bits_shared=4, shared_gate=1,
                         layers=40, seed=0x5EED0004)

# 62-layer stack, mixed bits: 4-bit gate/up, 6-bit down, two ungated shared experts.
DOTS_MIXED_STACK = Shape("dots.llm1-like stack, 62 layers, 4/4/6-bit, two shared experts",
                         din=4096, dff=1408, n_experts=128, top_k=6, bits_gate=4, bits_up=4,
                         bits_down=6, n_shared=2, dff_shared=1408, bits_shared=4, shared_gate=0,
                         layers=62, seed=0x5EED0005)

ALL = {
    "qwen3_layer_4bit": QWEN3_30B_A3B_4BIT_LAYER,
    "qwen15_layer_shared": QWEN15_MOE_A27B_LAYER,
    "qwen3_stack_8bit": QWEN3_30B_A3B_8BIT_STACK,
    "e512_stack": E512_TOP10_STACK,
    "dots_stack_mixed": DOTS_MIXED_STACK,
}


@dataclasses.dataclass(frozen=True)
class GemvShape:
    """A dense bf16 projection [n_out, n_in] of a decode token ("Measure attention projections
    instead of serving them, and record the amortisation trap": q/o and k/v of two models)."""
    name: str
    n_out: int
    n_in: int
    seed: int

    def weight_bytes(self) -> int:
        return self.n_out * self.n_in * 2


GEMV = {
    "qwen25_1p5b_qo": GemvShape("Qwen2.5-1.5B q/o projection, bf16", 1536, 1536, 0x5EED0101),
    "qwen25_1p5b_kv": GemvShape("Qwen2.5-1.5B k/v projection, bf16", 256, 1536, 0x5EED0102),
    "qwen3_8b_qo": GemvShape("Qwen3-8B q/o projection, bf16", 4096, 4096, 0x5EED0103),
    "qwen3_8b_kv": GemvShape("Qwen3-8B k/v projection, bf16", 1024, 4096, 0x5EED0104),
}
