"""Model shapes and decode workloads used across tests and the benchmark.

The shapes follow the Llama-style dense decoder family that the persistent
decode megakernel pages target (AutoMegaKernel explainer, "Methodology":
HuggingFace Llama-family models; Kog monokernel tutorial: an FP16 2B model at
batch 1).  No trained checkpoints exist here, so every workload is a seeded
random model with the stated shapes; weights ~ N(0, 0.02) rounded to the
storage type, norm gains 1.
"""
from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ffn: int
    vocab: int
    seed: int
    prompt_len: int
    decode_steps: int
    wdtype: str = "bf16"          # storage type of the GEMV weights: bf16 | fp16 | int8 | int4 | fp8
    rms_eps: float = 1e-5
    rope_theta: float = 1e4
    base_dtype: str = "bf16"      # storage type the random weights are drawn into

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def max_seq(self) -> int:
        return self.prompt_len + self.decode_steps

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    # 2 layers, d 256, 4 q / 2 kv heads of 64, FFN 768, vocab 512; prompt 8, decode 32.
    "tiny": Workload("tiny", 2, 256, 4, 2, 64, 768, 512, seed=0, prompt_len=8, decode_steps=32),
    # ~1B: 16 layers, d 2048, 32 q / 8 kv heads of 64, FFN 8192, vocab 32000, untied head.
    "llama-1b": Workload("llama-1b", 16, 2048, 32, 8, 64, 8192, 32000, seed=1,
                         prompt_len=128, decode_steps=256),
    # ~2B fp16: 24 layers, d 2560, 20 q / 4 kv heads of 128, FFN 6912, vocab 32000.
    "llama-2b-fp16": Workload("llama-2b-fp16", 24, 2560, 20, 4, 128, 6912, 32000, seed=2,
                              prompt_len=512, decode_steps=512, wdtype="fp16", base_dtype="fp16"),
    # The 1B model (seed 1 weights) with weight-only quantised GEMVs.
    "llama-1b-int8": Workload("llama-1b-int8", 16, 2048, 32, 8, 64, 8192, 32000, seed=1,
                              prompt_len=128, decode_steps=256, wdtype="int8"),
    "llama-1b-int4": Workload("llama-1b-int4", 16, 2048, 32, 8, 64, 8192, 32000, seed=1,
                              prompt_len=128, decode_steps=256, wdtype="int4"),
    # The same model with FP8 E4M3 GEMV weights, one fp16 scale per 128 k.
    "llama-1b-fp8": Workload("llama-1b-fp8", 16, 2048, 32, 8, 64, 8192, 32000, seed=1,
                             prompt_len=128, decode_steps=256, wdtype="fp8"),
    # Llama-3-8B shape, 8192-token prefilled KV cache, decode 128.
    "llama3-8b-8k": Workload("llama3-8b-8k", 32, 4096, 32, 8, 128, 14336, 128256, seed=4,
                             prompt_len=8192, decode_steps=128, rope_theta=5e5),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]
