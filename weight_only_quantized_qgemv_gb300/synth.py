"""Seeded synthetic inputs for the quantized GEMV and the routed-expert MLP.

This module only draws random numbers with the distributions of the five
workloads (uniform codes, lognormal or power-of-two group scales, N(0,1)
activations, top-k routing with softmax router weights).  It holds none of the
method's arithmetic: a packed buffer is drawn directly as random bytes, which is
exactly "uniform codes" for every format because each byte holds whole codes
(two int4/e2m1 nibbles, four int3 plane-A pairs, eight int3 plane-B bits).
The GPU path and the CPU oracle both read these buffers; neither lives here.

Layouts drawn (the library's ABI):
  int8 per row   [O][I] bytes, one f32 scale per row
  int4 grouped   [O][I/2] bytes (low nibble = even i), f32 scales [O][I/gs]
  int3-g64       plane A [O][I/4] then plane B [O][I/8] in one buffer,
                 f32 scales [O][I/64]
  MXFP4          [O][I/2] bytes of e2m1 nibbles, f32 scales [O][I/32]
  int4 per row   the int4 layout, one f32 scale per row
  int8 grouped   the int8 layout, f32 scales [O][I/gs]
  MXFP4 ue8m0    the MXFP4 layout, uint8 scale exponent bytes [O][I/32]
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# Format ids as colibri numbers its quantized storages (fmt 1, 2, 4, 5, 7, 8, 13).
INT8_ROW = 1
INT4_ROW = 2
INT4_G = 4
INT3_G64 = 5
MXFP4_G32 = 7
MXFP4_E8M0 = 8
INT8_G = 13

FMT_NAMES = {INT8_ROW: "int8_row", INT4_ROW: "int4_row", INT4_G: "int4_g", INT3_G64: "int3_g64",
             MXFP4_G32: "mxfp4_g32", MXFP4_E8M0: "mxfp4_e8m0", INT8_G: "int8_g"}


def fixed_group(fmt: int, I: int, gs: int | None = None) -> int:
    """Group size implied by a format (int8 per row: the whole row)."""
    if fmt in (INT8_ROW, INT4_ROW):
        return I
    if fmt == INT3_G64:
        return 64
    if fmt in (MXFP4_G32, MXFP4_E8M0):
        return 32
    return 32 if gs is None else gs


def packed_bytes(fmt: int, O: int, I: int) -> int:
    """Bytes of one packed [O][I] matrix."""
    if fmt in (INT8_ROW, INT8_G):
        return O * I
    if fmt in (INT4_ROW, INT4_G, MXFP4_G32, MXFP4_E8M0):
        return O * I // 2
    if fmt == INT3_G64:
        return O * I // 4 + O * I // 8
    raise ValueError(f"unknown fmt {fmt}")


def scale_itemsize(fmt: int) -> int:
    """Bytes of one stored scale: one ue8m0 byte, else an f32."""
    return 1 if fmt == MXFP4_E8M0 else 4


def generator(seed: int, *spawn_key: int) -> np.random.Generator:
    """PCG64 stream for (seed, spawn_key...); independent streams per key."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=tuple(spawn_key))))


def draw_packed(fmt: int, O: int, I: int, rng: np.random.Generator) -> np.ndarray:
    """Packed weights with uniform codes (int8: uniform in [-127, 127]).

    Uniform codes in every nibble, pair or bit are uniform bytes, which come
    straight from the generator's raw 64-bit output.
    """
    if fmt in (INT8_ROW, INT8_G):
        return rng.integers(-127, 128, size=O * I, dtype=np.int8).view(np.uint8)
    n = packed_bytes(fmt, O, I)
    raw = rng.bit_generator.random_raw((n + 7) // 8).view(np.uint8)
    return raw[:n].copy() if n % 8 else raw


def draw_scales(O: int, I: int, gs: int, rng: np.random.Generator, kind: str,
                mu: float = -4.0, sigma: float = 0.5, fmt: int | None = None) -> np.ndarray:
    """f32 scales [O][I/gs]: 'lognormal' (mu, sigma) or 'pow2' (2^k, k uniform in [-8, 0]).

    fmt=MXFP4_E8M0 draws the stored exponent bytes 127 + k instead: k uniform
    in [-8, 0] ('pow2'), or k = round(log2 of a lognormal(mu, sigma) draw).
    """
    n = O * (I // gs)
    if fmt == MXFP4_E8M0:
        if kind == "pow2":
            k = rng.integers(-8, 1, size=n)
        elif kind == "lognormal":
            z = rng.standard_normal(size=n)
            k = np.rint((z * sigma + mu) / np.log(2.0)).astype(np.int64)
        else:
            raise ValueError(kind)
        return (127 + k).astype(np.uint8)
    if kind == "lognormal":
        z = rng.standard_normal(size=n, dtype=np.float32)
        return np.exp(z * np.float32(sigma) + np.float32(mu)).astype(np.float32)
    if kind == "pow2":
        return np.ldexp(np.ones(n, dtype=np.float32), rng.integers(-8, 1, size=n)).astype(np.float32)
    raise ValueError(kind)


def draw_x(s: int, I: int, rng: np.random.Generator) -> np.ndarray:
    """Activations x f32 [s][I], N(0, 1)."""
    return rng.standard_normal(size=(s, I), dtype=np.float32)


def draw_routing(s: int, k: int, E: int, rng: np.random.Generator):
    """Per token: k distinct experts drawn uniformly, router weights = softmax of k N(0,1) logits.

    The router itself runs on the host in the engines the pages describe; here it
    is replaced by these draws, which the workloads fix.
    """
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(s)]).astype(np.int32)
    logits = rng.standard_normal(size=(s, k))
    w = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids.reshape(s, k), w.reshape(s, k)


# ---------------------------------------------------------------------------
# The five workloads (seed = 1000 + workload index).
# ---------------------------------------------------------------------------

@dataclass
class GemvWorkload:
    name: str
    fmt: int
    O: int
    I: int
    s: int
    gs: int
    scale_kind: str
    scale_mu: float
    seed: int
    x_key: int = 0
    gemm: bool = False      # a prefill batch, run through the tensor-core GEMM

    @property
    def weight_bytes(self) -> int:
        return packed_bytes(self.fmt, self.O, self.I)

    @property
    def scale_bytes(self) -> int:
        return scale_itemsize(self.fmt) * self.O * (self.I // self.gs)

    def weights(self, copy: int = 0):
        """(packed uint8, scales f32 or ue8m0 bytes) for weight copy `copy` (copies differ, same law)."""
        rng = generator(self.seed, 1, copy)
        w = draw_packed(self.fmt, self.O, self.I, rng)
        sc = draw_scales(self.O, self.I, self.gs, rng, self.scale_kind, self.scale_mu, fmt=self.fmt)
        return w, sc

    def x(self):
        return draw_x(self.s, self.I, generator(self.seed, 2, self.x_key))


@dataclass
class ExpertWorkload:
    name: str
    fmt: int
    E: int
    D: int
    F: int
    s: int
    k: int
    gs: int
    scale_kind: str
    scale_mu: float
    seed: int
    _cache: dict = field(default_factory=dict, repr=False)

    # Matrix ids inside one expert.
    GATE, UP, DOWN = 0, 1, 2

    def matrix_shape(self, which: int):
        return (self.F, self.D) if which in (self.GATE, self.UP) else (self.D, self.F)

    def expert_bytes(self) -> int:
        """Packed + scale bytes of one expert's three matrices."""
        tot = 0
        for which in (self.GATE, self.UP, self.DOWN):
            O, I = self.matrix_shape(which)
            tot += packed_bytes(self.fmt, O, I) + scale_itemsize(self.fmt) * O * (I // self.gs)
        return tot

    def expert_matrix(self, e: int, which: int):
        """(packed, scales) of expert e's gate/up/down, drawn from its own stream."""
        O, I = self.matrix_shape(which)
        rng = generator(self.seed, 10, e, which)
        w = draw_packed(self.fmt, O, I, rng)
        sc = draw_scales(O, I, self.gs, rng, self.scale_kind, self.scale_mu, fmt=self.fmt)
        return w, sc

    MATRICES = (("gate", 0), ("up", 1), ("down", 2))

    def sizes(self, which: int):
        """(packed bytes, scale count) of one expert matrix."""
        O, I = self.matrix_shape(which)
        return packed_bytes(self.fmt, O, I), O * (I // self.gs)

    def generate(self, experts, sink, threads: int = 16):
        """Draw the given experts' matrices in parallel, calling
        sink(name, slot, packed, scales) for each (slot = position in `experts`)."""
        from concurrent.futures import ThreadPoolExecutor
        experts = [int(e) for e in experts]

        def one(job):
            slot, e, name, which = job
            w, sc = self.expert_matrix(e, which)
            sink(name, slot, w, sc)

        jobs = [(slot, e, name, which) for name, which in self.MATRICES for slot, e in enumerate(experts)]
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, jobs))

    def store(self, experts=None, threads: int = 16):
        """{gate, gate_s, up, up_s, down, down_s}: the given experts (all by
        default) back to back, in host memory."""
        experts = list(range(self.E)) if experts is None else [int(e) for e in experts]
        out = {}
        for name, which in self.MATRICES:
            nb, ns = self.sizes(which)
            out[name] = np.empty(len(experts) * nb, dtype=np.uint8)
            out[name + "_s"] = np.empty(len(experts) * ns, dtype=np.uint8 if self.fmt == MXFP4_E8M0 else np.float32)

        def sink(name, slot, w, sc):
            nb, ns = w.size, sc.size
            out[name][slot * nb:(slot + 1) * nb] = w
            out[name + "_s"][slot * ns:(slot + 1) * ns] = sc

        self.generate(experts, sink, threads)
        return out

    def x(self, step: int = 0):
        return draw_x(self.s, self.D, generator(self.seed, 2, step))

    def routing(self, step: int = 0):
        return draw_routing(self.s, self.k, self.E, generator(self.seed, 3, step))

    def router_logits(self, step: int = 0):
        """Router logits [s][E], N(0, 1), for routing on the device (top-k of them is k
        experts drawn uniformly without replacement, as in routing())."""
        return generator(self.seed, 5, step).standard_normal(size=(self.s, self.E), dtype=np.float32)


def workload(name: str):
    """The named workload.  Names state format, sizes and batch."""
    table = {
        # int8 per row, 1024 x 1024, s = 1; row scales lognormal(-5, 0.5).
        "int8_row_1024x1024_s1": GemvWorkload("int8_row_1024x1024_s1", INT8_ROW, 1024, 1024, 1, 1024,
                                               "lognormal", -5.0, 1001),
        # int4 group 32, O = 16384, I = 6144, s = 1 and s = 4; scales lognormal(-4, 0.5).
        "int4_g32_16384x6144_s1": GemvWorkload("int4_g32_16384x6144_s1", INT4_G, 16384, 6144, 1, 32,
                                                "lognormal", -4.0, 1002),
        "int4_g32_16384x6144_s4": GemvWorkload("int4_g32_16384x6144_s4", INT4_G, 16384, 6144, 4, 32,
                                                "lognormal", -4.0, 1002, x_key=4),
        # int3-g64 dual plane, O = 6144, I = 16384 (o_proj-like long rows), s = 1.
        "int3_g64_6144x16384_s1": GemvWorkload("int3_g64_6144x16384_s1", INT3_G64, 6144, 16384, 1, 64,
                                                "lognormal", -4.0, 1003),
        # MXFP4 expert MLP, one token, top-8 of 256 experts; scales 2^k, k in [-8, 0].
        "mxfp4_experts_E256_D6144_F2048_s1_k8": ExpertWorkload("mxfp4_experts_E256_D6144_F2048_s1_k8",
                                                               MXFP4_G32, 256, 6144, 2048, 1, 8, 32,
                                                               "pow2", 0.0, 1004),
        # int4-g32 expert group, 8 tokens, top-8 of 256 experts each.
        "int4_g32_experts_E256_D6144_F2048_s8_k8": ExpertWorkload("int4_g32_experts_E256_D6144_F2048_s8_k8",
                                                                  INT4_G, 256, 6144, 2048, 8, 8, 32,
                                                                  "lognormal", -4.0, 1005),
        # Storage variants of the same decoders: int4 with one scale per row,
        # int8 with one scale per 64 inputs, and the MXFP4 expert workload with
        # its scales as ue8m0 exponent bytes (same seed and exponent draws as
        # the f32 one above, so the two hold the same values).
        "int4_row_16384x6144_s1": GemvWorkload("int4_row_16384x6144_s1", INT4_ROW, 16384, 6144, 1, 6144,
                                                "lognormal", -6.0, 1006),
        "int8_g64_16384x6144_s1": GemvWorkload("int8_g64_16384x6144_s1", INT8_G, 16384, 6144, 1, 64,
                                                "lognormal", -7.0, 1007),
        "mxfp4_e8m0_experts_E256_D6144_F2048_s1_k8": ExpertWorkload("mxfp4_e8m0_experts_E256_D6144_F2048_s1_k8",
                                                                    MXFP4_E8M0, 256, 6144, 2048, 1, 8, 32,
                                                                    "pow2", 0.0, 1004),
        # Prefill batches through the tensor-core GEMM: the int4-g32 matrix with
        # 512 activation rows (the pages' prefill measurements use 512-row
        # prompts) and with 32 (the engines' default prefill chunk).
        "int4_g32_16384x6144_s512_prefill": GemvWorkload("int4_g32_16384x6144_s512_prefill", INT4_G, 16384, 6144,
                                                         512, 32, "lognormal", -4.0, 1002, x_key=512, gemm=True),
        "int4_g32_16384x6144_s32_prefill": GemvWorkload("int4_g32_16384x6144_s32_prefill", INT4_G, 16384, 6144,
                                                        32, 32, "lognormal", -4.0, 1002, x_key=32, gemm=True),
    }
    return table[name]


WORKLOADS = [
    "int8_row_1024x1024_s1",
    "int4_g32_16384x6144_s1",
    "int4_g32_16384x6144_s4",
    "int3_g64_6144x16384_s1",
    "mxfp4_experts_E256_D6144_F2048_s1_k8",
    "int4_g32_experts_E256_D6144_F2048_s8_k8",
]

# Workloads of the storage variants (measured like the ones above, not part of
# the default set).
VARIANT_WORKLOADS = [
    "int4_row_16384x6144_s1",
    "int8_g64_16384x6144_s1",
    "mxfp4_e8m0_experts_E256_D6144_F2048_s1_k8",
]

# Prefill workloads (the tensor-core GEMM).
PREFILL_WORKLOADS = [
    "int4_g32_16384x6144_s512_prefill",
    "int4_g32_16384x6144_s32_prefill",
]
