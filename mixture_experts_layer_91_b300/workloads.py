"""Layer shapes of the synthetic workloads (no arithmetic of the method here).

Each workload is one MoE layer: T tokens of width d, K_s shared experts
always active, N_r routed experts of which top_k are selected per token, all
experts SwiGLU FFNs of intermediate width I.

The shapes follow the model sizes the DeepSeekMoE release note
(aibard123.com, "multi-scale models") and the DeepSeekMoE translation
(gitcode.csdn.net, section 3.1: mN fine-grained experts, mK active) describe:
a 2B model with 1 shared + 63 routed experts (top-7), a 16B model with
2 shared + 64 routed (top-6), a 145B model with 4 shared + 128 routed
(top-12), and a GShard-style coarse layer (16 experts, noisy top-2, the
gate of the "Outrageously Large Neural Networks" notes on
blog.carolineworld.cn, section 2).
"""

from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    n_routed: int
    n_shared: int
    top_k: int
    d_ff: int
    renormalize: bool = False
    noisy: bool = False
    bias: bool = False          # auxiliary-loss-free selection bias
    fp32: bool = False          # activations and expert weights in fp32 (else bf16)
    seed: int = 91
    capacity: int = 0           # assignments an expert accepts (0 = dropless)
    act: str = "swiglu"         # expert FFN: "swiglu" or GShard's "relu" (no W3)
    combine: str = "rows"       # bf16 combine: "rows" (bf16 expert rows + combine kernel) or "scatter"

    @property
    def n_experts(self) -> int:
        return self.n_routed + self.n_shared

    @property
    def n_assign(self) -> int:
        return self.T * self.top_k

    @property
    def n_mats(self) -> int:
        """d x I weight matrices per expert: W1, W3, W2 (SwiGLU) or W1, W2 (ReLU)."""
        return 2 if self.act == "relu" else 3

    def flops(self) -> float:
        """Algorithmic FLOPs of one forward: the router x.W_g (twice with the
        noise projection) plus one d x I product per weight matrix per active
        expert per token (dropless)."""
        router = 2.0 * self.T * self.d * self.n_routed * (2 if self.noisy else 1)
        ffn = 2.0 * self.n_mats * self.T * self.d * self.d_ff * (self.top_k + self.n_shared)
        return router + ffn

    def with_tokens(self, T: int, name: str | None = None) -> "Workload":
        return replace(self, T=T, name=name or f"{self.name}_T{T}")


TINY_FP32 = Workload("tiny_fp32_T256", T=256, d=128, n_routed=16, n_shared=1,
                     top_k=4, d_ff=64, fp32=True, seed=91)
DSMOE_2B = Workload("dsmoe2b_T8192", T=8192, d=1280, n_routed=63, n_shared=1,
                    top_k=7, d_ff=896, seed=92)
DSMOE_16B = Workload("dsmoe16b_T16384", T=16384, d=2048, n_routed=64, n_shared=2,
                     top_k=6, d_ff=1408, seed=93)
GSHARD_NOISY = Workload("gshard_noisy_top2_T16384", T=16384, d=2048, n_routed=16,
                        n_shared=0, top_k=2, d_ff=5632, renormalize=True, noisy=True,
                        seed=94)
DSMOE_145B = Workload("dsmoe145b_prefill_T32768", T=32768, d=4096, n_routed=128,
                      n_shared=4, top_k=12, d_ff=1024, bias=True, seed=95)
DSMOE_145B_DECODE = replace(DSMOE_145B, name="dsmoe145b_decode_T64", T=64)

# GShard's own expert form wo.ReLU(wi.x) on the GShard-style layer (same
# parameters per expert as its SwiGLU twin minus W3), with a Switch-style
# expert capacity of 1.25 x the mean load: ceil(1.25 * T * k / E).
GSHARD_RELU_CAP = replace(GSHARD_NOISY, name="gshard_relu_cap1.25_T16384", act="relu",
                          capacity=-(-5 * 16384 * 2 // (4 * 16)), seed=96)

# The headline layer with the down projection's gate-weighted scatter-add into
# an fp32 accumulator (moe_combine_mode MOE_COMBINE_SCATTER_ADD) instead of
# stored bf16 expert rows; same inputs.
DSMOE_16B_SCATTER = replace(DSMOE_16B, name="dsmoe16b_scatter_T16384", combine="scatter")

ALL = [TINY_FP32, DSMOE_2B, DSMOE_16B, GSHARD_NOISY, DSMOE_145B, DSMOE_145B_DECODE, GSHARD_RELU_CAP,
       DSMOE_16B_SCATTER]
BY_NAME = {w.name: w for w in ALL}

# the layer the throughput headline is quoted on: the 16B-shaped layer at 16K tokens
HEADLINE = DSMOE_16B
