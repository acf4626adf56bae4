"""Decode-projection workloads: shapes of a Llama-3.1-8B-shaped model (random
init, shapes only) and the device-resident decode step built from them.

One decode step at batch 1 multiplies, in every layer, the hidden vector by the
fused Q/K/V projection (4,096 + 1,024 + 1,024 rows), the output projection
(4,096 rows), the fused gate/up projection (14,336 + 14,336 rows) and the down
projection (4,096 rows over K = 14,336), then the LM head (128,256 rows)
("Decode GEMV at half of HBM bandwidth", causes 1 and 3; "GPU performance
chains", "Launch gaps in a decode step"). The projections are not chained: with
random weights and no nonlinearity in between, each layer reads its own
activation vector x4096_l (shared by QKV, o_proj and gate/up) and x14336_l
(read by down); the LM head reads its own x. Each projection group is one
launch: 4 per layer plus the LM head, 129 for 32 layers, captured as one graph.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding, inputs, roofline

LLAMA_8B = dict(layers=32, hidden=4096, intermediate=14336, vocab=128256, q_rows=4096, kv_rows=1024)

# Single-projection shapes (N, K) of that model.
SHAPES = {
    "k_proj": (1024, 4096),
    "down_proj": (4096, 14336),
    "qkv": (6144, 4096),
    "o_proj": (4096, 4096),
    "gate_up": (28672, 4096),
    "lm_head": (128256, 4096),
}

# Ragged shapes with ldw = K rounded up to a multiple of 8.
TAILS = [(7, 129), (4097, 4103), (1, 8191), (33, 65537)]


def decode_step_spec(**overrides) -> dict:
    spec = dict(LLAMA_8B)
    spec.update(overrides)
    return spec


@dataclass
class Proj:
    name: str
    W: torch.Tensor          # BF16 weights, or the INT4 / FP8 codes
    x: torch.Tensor
    y: torch.Tensor
    N: int
    K: int
    ldw: int                 # row stride (elements for BF16, bytes for codes)
    group: int
    S: torch.Tensor | None = None   # INT4 group scales / FP8 row scales
    lds: int = 0


WEIGHT_KINDS = {"bf16": binding.GEMV_WEIGHT_BF16, "int4": binding.GEMV_WEIGHT_INT4,
                "fp8": binding.GEMV_WEIGHT_FP8}


class DecodeStep:
    """Device-resident weights, activations and outputs of one decode step, with
    BF16, INT4 (128-column groups, BF16 scales) or FP8 (E4M3, FP32 row scales)
    weights."""

    def __init__(self, spec: dict, seed: int = 0, device="cuda", weights: str = "bf16", batch: int = 1):
        if weights not in WEIGHT_KINDS:
            raise ValueError(f"weights must be one of {sorted(WEIGHT_KINDS)}")
        if not 1 <= batch <= binding.GEMV_MAX_BATCH:
            raise ValueError("batch must be 1..16")
        self.spec = spec
        self.device = device
        self.weights = weights
        self.batch = batch
        self.projs: list[Proj] = []
        self.xs: list[tuple[torch.Tensor, int]] = []
        H, I, V = spec["hidden"], spec["intermediate"], spec["vocab"]
        Q, KV = spec["q_rows"], spec["kv_rows"]
        L = spec["layers"]
        # Every activation vector lives in one buffer and every output in
        # another (views at 16-byte multiples), so a step's inputs and outputs
        # each cross the host link as one copy (gemv_plan_launch_host_io).
        self.x_arena = torch.empty(batch * (L * (H + I) + H), dtype=torch.bfloat16, device=device)
        self.y_arena = torch.empty(batch * (L * (Q + 2 * KV + H + 2 * I + H) + V), dtype=torch.float32,
                                   device=device)
        self._x_off = 0
        self._y_off = 0
        group = 0
        for l in range(spec["layers"]):
            base = 16 * l
            xh = self._x_view(inputs.activations(batch, H, seed=seed, index=base + 14, device=device))
            xi = self._x_view(inputs.activations(batch, I, seed=seed, index=base + 15, device=device))
            self.xs += [(xh, base + 14), (xi, base + 15)]
            group += 1
            for j, (nm, n) in enumerate([("q", Q), ("k", KV), ("v", KV)]):
                self._add(f"l{l}.{nm}_proj", n, H, xh, group, seed, base + j)
            self._add(f"l{l}.o_proj", H, H, xh, 0, seed, base + 3)
            group += 1
            self._add(f"l{l}.gate_proj", I, H, xh, group, seed, base + 4)
            self._add(f"l{l}.up_proj", I, H, xh, group, seed, base + 5)
            self._add(f"l{l}.down_proj", H, I, xi, 0, seed, base + 6)
        base = 16 * spec["layers"]
        xl = self._x_view(inputs.activations(batch, H, seed=seed, index=base + 1, device=device))
        self.xs.append((xl, base + 1))
        self._add("lm_head", V, H, xl, 0, seed, base)
        assert self._x_off == self.x_arena.numel() and self._y_off == self.y_arena.numel()

    def _x_view(self, x: torch.Tensor) -> torch.Tensor:
        B, n = x.shape
        v = self.x_arena[self._x_off:self._x_off + B * n].view(B, n)
        v.copy_(x)
        self._x_off += B * n
        return v

    def _add(self, name, N, K, x, group, seed, index):
        y = self.y_arena[self._y_off:self._y_off + self.batch * N].view(self.batch, N)
        self._y_off += self.batch * N
        if self.weights == "bf16":
            ldw = inputs.padded_ldw(K)
            W = inputs.weight(N, K, ldw, seed=seed, index=index, device=self.device)
            self.projs.append(Proj(name, W, x, y, N, K, ldw, group))
        elif self.weights == "fp8":
            W, S = inputs.fp8_weight(N, K, seed=seed, index=index, device=self.device)
            self.projs.append(Proj(name, W, x, y, N, K, W.shape[1], group, S, 0))
        else:
            W, S = inputs.w4_weight_device(N, K, seed=seed, index=index, device=self.device)
            self.projs.append(Proj(name, W, x, y, N, K, W.shape[1], group, S, S.shape[1]))

    def plan(self, rms_eps: float | None = None, streamk: bool = False) -> binding.Plan:
        """The step as one plan. With rms_eps, the projections that read a
        normalised activation in the model (QKV, gate/up and the LM head) take
        the RMSNorm prologue; o_proj and down read the raw one. With streamk,
        every launch runs the stream-K kernel."""
        def eps_of(p):
            if rms_eps is None:
                return None
            return rms_eps if (p.name.endswith(("q_proj", "k_proj", "v_proj", "gate_proj", "up_proj"))
                               or p.name == "lm_head") else None
        kind = WEIGHT_KINDS[self.weights]
        return binding.Plan([(p.W, p.x, p.y, p.N, p.K, p.ldw, self.batch, p.group, eps_of(p), streamk, kind, p.S,
                              p.lds) for p in self.projs], keepalive=self)

    def outputs(self):
        return [p.y for p in self.projs]

    def refresh_x(self, seed: int) -> None:
        """Overwrite every activation vector in place (the plan keeps its addresses)."""
        for x, index in self.xs:
            x.copy_(inputs.activations(self.batch, x.shape[1], seed=seed, index=index, device=self.device))

    def checks(self):
        for p in self.projs:
            yield p.name, p.W, p.x, p.y, p.K

    def _wbytes(self, p) -> int:
        """Weight bytes of one projection: BF16 2*N*K; INT4 N*K/2 codes plus
        2*N*K/128 scale bytes; FP8 N*K codes plus 4*N scale bytes."""
        if self.weights == "bf16":
            return 2 * p.N * p.K
        if self.weights == "fp8":
            return p.N * p.K + 4 * p.N
        return p.N * p.K // 2 + 2 * p.N * (p.K // inputs.W4_GROUP)

    def algorithmic_bytes(self) -> int:
        """Sum of weight bytes + B*K*2 + B*N*4 over the projections; a fused
        launch moves its x once, so each launch group counts x once."""
        total = 0
        seen_groups = set()
        for p in self.projs:
            total += self._wbytes(p) + 4 * self.batch * p.N
            if p.group == 0 or p.group not in seen_groups:
                total += 2 * self.batch * p.K
                seen_groups.add(p.group)
        return total

    def weight_bytes(self) -> int:
        return sum(self._wbytes(p) for p in self.projs)


def step_bytes_formula(spec: dict, batch: int = 1) -> int:
    """Algorithmic bytes of the step at `batch` rows of x, with fused groups
    counted as one GEMV each (QKV 6,144 rows; gate/up 28,672 rows)."""
    H, I, V = spec["hidden"], spec["intermediate"], spec["vocab"]
    Q, KV = spec["q_rows"], spec["kv_rows"]
    B = batch
    layer = (roofline.algorithmic_bytes(Q + 2 * KV, H, B) + roofline.algorithmic_bytes(H, H, B)
             + roofline.algorithmic_bytes(2 * I, H, B) + roofline.algorithmic_bytes(H, I, B))
    return spec["layers"] * layer + roofline.algorithmic_bytes(V, H, B)
