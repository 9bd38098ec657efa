"""Seeded synthetic inputs for the sparse MoE FFN layer.

This module is the one thing the GPU library's callers and the fp64 oracle's
callers share: it draws random tensors and names the workload shapes.  It holds
none of the layer's arithmetic (no scores, no selection, no FFN), only random
numbers with the stated distributions.

Workloads (shapes and distributions; names by what they are):

  tiny_f32            T=64, d=256, E=8, K=2, I=512, no shared expert, fp32.
                      x ~ N(0,1); router and expert weights ~ N(0, 1/d).
  mixtral_prefill     T=4096, d=4096, E=8, K=2, I=14336, no shared expert, bf16.
                      x ~ N(0,1); w_g, w_gate, w_up ~ N(0, 1/d); w_down ~ N(0, 1/I).
  dsv3_decode         T=8, d=7168, E=256, K=8, I=2048, one shared expert Is=2048, bf16.
                      x ~ N(0,1); all weights ~ N(0, 1/d).
  dsv3_prefill_zipf   T=16384, otherwise dsv3_decode shapes, plus a per-expert bias
                      b_e = -s * beta * ln(r_e) on the router scores, r a seeded
                      permutation of 1..E, s = 1.2, beta = ZIPF_BETA, so expert
                      popularity falls off like a Zipf law in rank.
  dsv3_sweep_T{n}     dsv3_decode shapes at T = n, n in {1, 8, 64, 512, 4096}.
  dsv3_decode_sigmoid dsv3_decode with the DeepSeek-V3 router (sigmoid affinities,
                      weights a / (sum a + 1e-6)).
  dsv3_decode_fp8     dsv3_decode with 8-bit expert weights (routed and shared):
  mixtral_prefill_fp8 mixtral_prefill likewise (dsv3_decode_fp8_E32: the decode
                      layer with a pool of 32 experts).  Each weight is an E4M3 code drawn
                      as random bits -- sign uniform, exponent field uniform in
                      9..15, mantissa uniform, the NaN pattern S.1111.111 redrawn
                      as S.1111.110 -- so magnitudes are log-uniform over [4, 448]
                      with an RMS of about 162; each weight row has its own fp32
                      scale std / 162 * U(0.8, 1.2), std being the bf16 workload's
                      weight std.  The router weights stay bf16.
  mixtral_prefill_w8a8, dsv3_sweep_w8a8_T{512,4096}, dsv3_decode_w8a8,
  dsv3_prefill_zipf_w8a8
                      the 8-bit-weight workloads run with 8-bit activations too
                      (the library quantises x and the hidden rows per row).

Every tensor has its own sub-seed, splitmix64(seed ^ fnv1a64(name)), so adding
or resizing one tensor never changes another.  Large weights are drawn one
expert at a time from a single generator (deterministic for a given device
type and torch build), on whatever device the caller names.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

MASK64 = (1 << 64) - 1
ZIPF_S = 1.2
# Scale of the log-rank bias (in units of the router score's standard deviation,
# which is 1 for x ~ N(0,1) and w_g ~ N(0,1/d)).  With top-8 of 256 experts this
# gives a log-log slope of the sorted expert counts near -1.2 over ranks 1..64 and
# a hottest expert with more than 10x the mean count (checked by a test).
ZIPF_BETA = 0.65


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    d: int
    E: int
    K: int
    I: int
    Is: int = 0           # 0 = no shared expert
    dtype: str = "bf16"   # "bf16" or "f32"
    down_std: str = "d"   # "d": w_down ~ N(0,1/d); "inter": N(0,1/I)
    zipf_bias: bool = False
    router: str = "softmax"   # "softmax" or "sigmoid" (DeepSeek-V3 affinities)
    weights: str = "act"      # "act": experts in dtype; "e4m3": 8-bit codes + row scales;
                              # "e4m3b": 8-bit codes + one scale per 128 x 128 block
    acts: str = "act"         # "e4m3": the experts' input and hidden rows quantised (W8A8)
    seed: int = 0
    extra: dict = field(default_factory=dict, compare=False)

    def with_T(self, T: int) -> "LayerConfig":
        return replace(self, T=T, name=f"{self.name}@T{T}")


CONFIGS: dict[str, LayerConfig] = {
    "tiny_f32": LayerConfig("tiny_f32", T=64, d=256, E=8, K=2, I=512, Is=0, dtype="f32"),
    "mixtral_prefill": LayerConfig("mixtral_prefill", T=4096, d=4096, E=8, K=2, I=14336, Is=0,
                                   dtype="bf16", down_std="inter"),
    "dsv3_decode": LayerConfig("dsv3_decode", T=8, d=7168, E=256, K=8, I=2048, Is=2048),
    "dsv3_prefill_zipf": LayerConfig("dsv3_prefill_zipf", T=16384, d=7168, E=256, K=8, I=2048,
                                     Is=2048, zipf_bias=True),
}
# DeepSeek-V3 decode with its own router: sigmoid affinities, weights a / (sum a + 1e-6)
CONFIGS["dsv3_decode_sigmoid"] = LayerConfig("dsv3_decode_sigmoid", T=8, d=7168, E=256, K=8,
                                             I=2048, Is=2048, router="sigmoid")
# 8-bit expert weights (E4M3 codes, one fp32 scale per weight row)
CONFIGS["dsv3_decode_fp8"] = replace(CONFIGS["dsv3_decode"], name="dsv3_decode_fp8",
                                     weights="e4m3")
CONFIGS["mixtral_prefill_fp8"] = replace(CONFIGS["mixtral_prefill"], name="mixtral_prefill_fp8",
                                         weights="e4m3")
for _t in (64, 512):
    CONFIGS[f"dsv3_sweep_fp8_T{_t}"] = replace(CONFIGS["dsv3_decode_fp8"],
                                               name=f"dsv3_sweep_fp8_T{_t}", T=_t)
# 8-bit expert weights with one fp32 scale per 128 x 128 block of each stacked
# matrix (DeepSeek-V3's checkpoint layout); the codes are those of the row-scaled
# configs above
CONFIGS["dsv3_decode_fp8b"] = replace(CONFIGS["dsv3_decode"], name="dsv3_decode_fp8b",
                                      weights="e4m3b")
CONFIGS["mixtral_prefill_fp8b"] = replace(CONFIGS["mixtral_prefill"], name="mixtral_prefill_fp8b",
                                          weights="e4m3b")
CONFIGS["dsv3_sweep_fp8b_T512"] = replace(CONFIGS["dsv3_decode_fp8b"], name="dsv3_sweep_fp8b_T512",
                                          T=512)
# the same block-scaled weights with 8-bit activations (x and h quantised per row)
CONFIGS["dsv3_decode_w8a8b"] = replace(CONFIGS["dsv3_decode_fp8b"], name="dsv3_decode_w8a8b",
                                       acts="e4m3")
CONFIGS["mixtral_prefill_w8a8b"] = replace(CONFIGS["mixtral_prefill_fp8b"],
                                           name="mixtral_prefill_w8a8b", acts="e4m3")
CONFIGS["dsv3_prefill_zipf_w8a8b"] = replace(CONFIGS["dsv3_prefill_zipf"],
                                             name="dsv3_prefill_zipf_w8a8b", weights="e4m3b",
                                             acts="e4m3")
# the same decode layer over a pool of 32 experts (1.4 GB of codes): small enough
# for multi-pass counter captures, still far larger than L2
CONFIGS["dsv3_decode_fp8_E32"] = replace(CONFIGS["dsv3_decode_fp8"], name="dsv3_decode_fp8_E32",
                                         E=32)
# the bf16 decode layer with a pool of 32 experts (2.8 GB of expert weights,
# still larger than L2): small enough for counter captures of the decode GEMMs
CONFIGS["dsv3_decode_E32"] = replace(CONFIGS["dsv3_decode"], name="dsv3_decode_E32", E=32)
# 8-bit weights and 8-bit activations (W8A8): the same weights; the library
# quantises x and h itself, so no extra tensor is drawn
CONFIGS["mixtral_prefill_w8a8"] = replace(CONFIGS["mixtral_prefill_fp8"],
                                          name="mixtral_prefill_w8a8", acts="e4m3")
for _t in (512, 4096):
    CONFIGS[f"dsv3_sweep_w8a8_T{_t}"] = replace(CONFIGS["dsv3_decode_fp8"],
                                                name=f"dsv3_sweep_w8a8_T{_t}", T=_t, acts="e4m3")
CONFIGS["dsv3_decode_w8a8"] = replace(CONFIGS["dsv3_decode_fp8"], name="dsv3_decode_w8a8",
                                      acts="e4m3")
# the T=4096 W8A8 per-expert shape (~128 rows per expert) over a pool of 64
# experts (2.8 GB of codes): small enough for counter captures
CONFIGS["dsv3_sweep_w8a8_T1024_E64"] = replace(CONFIGS["dsv3_sweep_w8a8_T4096"],
                                               name="dsv3_sweep_w8a8_T1024_E64", T=1024, E=64)
CONFIGS["dsv3_prefill_zipf_w8a8"] = replace(CONFIGS["dsv3_prefill_zipf"],
                                            name="dsv3_prefill_zipf_w8a8", weights="e4m3",
                                            acts="e4m3")
SWEEP_T = (1, 8, 64, 512, 4096)
for _t in SWEEP_T:
    CONFIGS[f"dsv3_sweep_T{_t}"] = LayerConfig(f"dsv3_sweep_T{_t}", T=_t, d=7168, E=256, K=8,
                                               I=2048, Is=2048)


def fnv1a64(s: str) -> int:
    h = 0xCBF29CE484222325
    for b in s.encode():
        h ^= b
        h = (h * 0x100000001B3) & MASK64
    return h


def splitmix64(z: int) -> int:
    z = (z + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def sub_seed(seed: int, name: str) -> int:
    # torch.Generator.manual_seed takes a 64-bit value; keep it non-negative 63-bit
    return splitmix64((seed & MASK64) ^ fnv1a64(name)) & ((1 << 63) - 1)


def _gen(device, seed: int, name: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(seed, name))
    return g


def torch_dtype(dtype: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]


def normal(shape, std: float, dtype: str, device, seed: int, name: str,
           chunk_dim0: bool = False) -> torch.Tensor:
    """N(0, std^2) samples in the storage dtype, drawn in fp32 and rounded once.

    With chunk_dim0 the tensor is drawn one leading index at a time (bounded
    temporary memory for the expert weight stacks)."""
    g = _gen(device, seed, name)
    out = torch.empty(shape, dtype=torch_dtype(dtype), device=device)
    if chunk_dim0:
        for i in range(shape[0]):
            out[i].copy_(torch.randn(shape[1:], generator=g, device=device,
                                     dtype=torch.float32).mul_(std))
    else:
        out.copy_(torch.randn(shape, generator=g, device=device, dtype=torch.float32).mul_(std))
    return out


def zipf_bias(E: int, seed: int, s: float = ZIPF_S, beta: float = ZIPF_BETA) -> torch.Tensor:
    """b_e = -s * beta * ln(r_e), r a seeded permutation of 1..E (fp32, CPU)."""
    g = _gen("cpu", seed, "zipf_rank")
    r = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    return (-s * beta * torch.log(r)).to(torch.float32)


E4M3_RMS = 162.0  # RMS of the code values drawn by e4m3_codes (162.13)


def e4m3_codes(shape, device, seed: int, name: str, chunk_dim0: bool = False) -> torch.Tensor:
    """Random E4M3 bit patterns (uint8): sign uniform, exponent field uniform in
    9..15, mantissa uniform, NaN (S.1111.111) replaced by S.1111.110."""
    g = _gen(device, seed, name)
    out = torch.empty(shape, dtype=torch.uint8, device=device)

    def draw(sh):
        e = torch.randint(9, 16, sh, generator=g, device=device, dtype=torch.int32)
        m = torch.randint(0, 8, sh, generator=g, device=device, dtype=torch.int32)
        sg = torch.randint(0, 2, sh, generator=g, device=device, dtype=torch.int32)
        m = torch.where((e == 15) & (m == 7), torch.full_like(m, 6), m)
        return (sg * 128 + e * 8 + m).to(torch.uint8)

    if chunk_dim0:
        for i in range(shape[0]):
            out[i].copy_(draw(tuple(shape[1:])))
    else:
        out.copy_(draw(tuple(shape)))
    return out


def row_scales(shape, std: float, device, seed: int, name: str) -> torch.Tensor:
    """One fp32 scale per weight row: std / E4M3_RMS * U(0.8, 1.2)."""
    g = _gen(device, seed, name)
    u = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    return (u * 0.4 + 0.8) * (std / E4M3_RMS)


def block_scales(rows: int, cols: int, std: float, device, seed: int, name: str) -> torch.Tensor:
    """One fp32 scale per 128 x 128 block of a stacked [rows][cols] matrix:
    [ceil(rows/128)][ceil(cols/128)], std / E4M3_RMS * U(0.8, 1.2)."""
    return row_scales(((rows + 127) // 128, (cols + 127) // 128), std, device, seed, name)


def is_fp8(cfg: LayerConfig) -> bool:
    """The expert matrices are E4M3 codes (row or block scales)."""
    return cfg.weights in ("e4m3", "e4m3b")


def make_weights(cfg: LayerConfig, device="cpu", only=None) -> dict:
    """Router, routed-expert and shared-expert weights, stored [out][in].

    For cfg.weights == "e4m3" the expert matrices are uint8 E4M3 codes and the
    dict also holds their row scales: s_gate, s_up [E][I], s_down [E][d] (ss_*
    for the shared expert); w_g stays in cfg.dtype.  For "e4m3b" the same
    codes with block scales over each stacked matrix: s_gate, s_up
    [E*I/128][d/128], s_down [E*d/128][I/128] (ss_* likewise).
    ``only`` (a set of names) draws just those tensors; each has its own
    sub-seed, so the values are the same as in a full draw."""
    d, E, I, Is, dt, sd = cfg.d, cfg.E, cfg.I, cfg.Is, cfg.dtype, cfg.seed
    std_d = 1.0 / math.sqrt(d)
    std_down = 1.0 / math.sqrt(I) if cfg.down_std == "inter" else std_d
    std_sdown = (1.0 / math.sqrt(Is) if cfg.down_std == "inter" else std_d) if Is else 0.0
    recipe = {
        "w_g": ((E, d), std_d, False),
        "w_gate": ((E, I, d), std_d, True),
        "w_up": ((E, I, d), std_d, True),
        "w_down": ((E, d, I), std_down, True),
    }
    if Is:
        recipe["ws_gate"] = ((Is, d), std_d, False)
        recipe["ws_up"] = ((Is, d), std_d, False)
        recipe["ws_down"] = ((d, Is), std_sdown, False)
    if is_fp8(cfg):
        out = {}
        for name, (shape, std, chunk) in recipe.items():
            sname = "s" + name[1:] if name.startswith("w_") else "ss" + name[2:]
            if name == "w_g":
                if only is None or name in only:
                    out[name] = normal(shape, std, dt, device, sd, name)
                continue
            if only is None or name in only:
                out[name] = e4m3_codes(shape, device, sd, name, chunk_dim0=chunk)
            if only is None or sname in only:
                if cfg.weights == "e4m3b":
                    rows = math.prod(shape[:-1])
                    out[sname] = block_scales(rows, shape[-1], std, device, sd, sname)
                else:
                    out[sname] = row_scales(shape[:-1], std, device, sd, sname)
        return out
    return {name: normal(shape, std, dt, device, sd, name, chunk_dim0=chunk)
            for name, (shape, std, chunk) in recipe.items() if only is None or name in only}


def make_x(cfg: LayerConfig, device="cpu", name: str = "x") -> torch.Tensor:
    return normal((cfg.T, cfg.d), 1.0, cfg.dtype, device, cfg.seed, name)


def make_bias(cfg: LayerConfig, device="cpu"):
    if not cfg.zipf_bias:
        return None
    return zipf_bias(cfg.E, cfg.seed).to(device)


def redraw_rows(x: torch.Tensor, rows, cfg: LayerConfig, attempt: int) -> torch.Tensor:
    """Replace the listed token rows of x with fresh N(0,1) draws from the
    sub-seed (seed, "x_redraw/<attempt>/<row>") (deterministic)."""
    x = x.clone()
    for r in rows:
        g = _gen(x.device, cfg.seed, f"x_redraw/{attempt}/{int(r)}")
        x[int(r)].copy_(torch.randn((cfg.d,), generator=g, device=x.device, dtype=torch.float32))
    return x


def grid_logits(T: int, E: int, seed: int, scale: int = 512, name: str = "logits",
                device="cpu") -> torch.Tensor:
    """Router scores on the grid round(N(0,1) * scale) / scale, exact in fp32.

    Distinct values differ by at least 1/scale (>= 1e-3 at scale 512); equal
    values occur and are decided only by the tie rule."""
    g = _gen(device, seed, name)
    z = torch.randn((T, E), generator=g, device=device, dtype=torch.float64)
    return (torch.round(z * scale) / scale).to(torch.float32)


def sample_tokens(T: int, n: int, seed: int, name: str = "sample") -> torch.Tensor:
    """A seeded sample of n distinct token ids in [0, T), sorted (int32, CPU)."""
    if n >= T:
        return torch.arange(T, dtype=torch.int32)
    g = _gen("cpu", seed, name)
    return torch.sort(torch.randperm(T, generator=g)[:n]).values.to(torch.int32)


def token_order(T: int, seed: int, name: str = "sample_order") -> torch.Tensor:
    """A seeded permutation of the token ids [0, T) (int64, CPU): the order in
    which a sampler that skips some tokens considers them."""
    g = _gen("cpu", seed, name)
    return torch.randperm(T, generator=g)


def to_host_array(t: torch.Tensor):
    """Host numpy view of a tensor for the oracle: bf16 -> uint16 bit patterns,
    fp32 -> float32, anything else as is."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
