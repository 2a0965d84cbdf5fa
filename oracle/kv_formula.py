"""KV-cache size in closed form (test infrastructure; see the package docstring).

Sources (page title, section):
  * "Ch. 6 Inference efficiency and serving", section 6.3 (the KV cache memory
    ledger): M_KV ~= 2 * L * B * T * H_kv * d_h * b, the leading 2 for keys
    and values; worked example L=32, B=1, T=8192, H_kv=8, d_h=128, b=2 gives
    2**30 bytes (1 GiB), 4 GiB with H_kv=32, 16 GiB / 64 GiB at B=16.
  * "LLM inference systems engineering", section 2.2.3: per token
    2 * h_kv * d_head * L * b = 131072 B (128 KiB) at h_kv=8, d_head=128,
    L=32, bf16; a 4096-token sequence is 512 MiB.
  * "The math of Transformer inference", section 5: 819,200 B per token for
    LLaMA-2-13B (L=40, K=40, H=128, bf16), 327,680 B for LLaMA-3-70B (L=80,
    K=8, H=128).
  * "LLM inference systems engineering", 2.4.2 (MLA): a latent cache stores
    (d_c + d_r) * L * b bytes per token -- 36,864 B (36 KiB) at d_c=512,
    d_r=64, L=32, bf16, 131072 / 36864 = 3.56 x less than the GQA case.
  * "The math of Transformer inference", MLA section: 61 x 576 x 2 = 70,272
    bytes per token for DeepSeek-V3; MHA with the same heads would store
    128 x (192 + 128) = 40,960 elements per layer, 71 x MLA's 576.
  * "Module 10: inference and serving", Lab 2: a 4-layer toy decoder with two
    KV heads of width 32 in float32 holds 555,008 bytes at 271 cached tokens,
    equal to 2*4*2*32*4*t.
"""


def kv_bytes(L: int, B: int, T: int, H_kv: int, d_h: int, b: int) -> int:
    """Bytes of K and V for L layers, B sequences of T cached tokens,
    H_kv KV heads of width d_h, b bytes per element."""
    return 2 * L * B * T * H_kv * d_h * b


def kv_bytes_per_token(L: int, H_kv: int, d_h: int, b: int) -> int:
    return kv_bytes(L, 1, 1, H_kv, d_h, b)


def paged_pool_bytes(num_blocks: int, block_size: int, H_kv: int, d_h: int, b: int,
                     L: int = 1) -> int:
    """Physical bytes of a paged pool of num_blocks blocks of block_size
    tokens: the same closed form with B*T replaced by the slots it holds."""
    return kv_bytes(L, 1, num_blocks * block_size, H_kv, d_h, b)


def mla_bytes_per_token(L: int, d_c: int, d_r: int, b: int) -> int:
    """Bytes per token of an MLA latent cache: the latent and the decoupled
    RoPE key of every layer."""
    return (d_c + d_r) * L * b
