"""Seeded synthetic inputs shaped like the models the pages train.

This module holds no arithmetic of the compression method. It only knows
tensor shapes and draws random numbers, so that the CUDA path and the CPU
oracle can be fed the very same bytes. Every draw comes from a
``torch.Generator`` seeded with ``1000*config + 100*learner + step``.

Model shapes stand in for the pages' workloads (no dataset or trained weights
are involved):

* ResNet-50 (161 parameter tensors, 25,557,032 values) -- the DGC page quotes
  its gradient as 97 MB (Deep Gradient Compression, Abstract).
* a 2-layer LSTM language model (hidden 1500, vocabulary 10,000) and a VGG-16
  convolution stack -- AdaComp's FC/recurrent and convolutional layers
  (AdaComp, Abstract).
* DeepSpeech-like GRU-sized tensors -- the 488 MB gradient of the DGC
  Abstract.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


# --------------------------------------------------------------------------
# model shapes
# --------------------------------------------------------------------------

def resnet50_shapes(width_div: int = 1) -> list[tuple[str, int]]:
    """Parameter tensors of ResNet-50 in definition order (torchvision naming).

    Stem 64x3x7x7 conv + BN, four bottleneck stages of [3, 4, 6, 3] blocks with
    widths 64/128/256/512 and expansion 4 (a 1x1 downsample conv + BN in the
    first block of each stage), then fc 1000x2048 + bias. ``width_div`` shrinks
    every channel count for small test cases while keeping the 161-tensor
    structure.
    """
    d = width_div
    out: list[tuple[str, int]] = []

    def conv(name, cout, cin, k):
        out.append((name + ".weight", (cout // d) * (cin // d if cin > 3 else cin) * k * k))

    def bn(name, c):
        out.append((name + ".weight", c // d))
        out.append((name + ".bias", c // d))

    conv("conv1", 64, 3, 7)
    bn("bn1", 64)
    cin = 64
    for li, (blocks, width) in enumerate(zip([3, 4, 6, 3], [64, 128, 256, 512]), start=1):
        for b in range(blocks):
            p = f"layer{li}.{b}"
            conv(p + ".conv1", width, cin, 1)
            bn(p + ".bn1", width)
            conv(p + ".conv2", width, width, 3)
            bn(p + ".bn2", width)
            conv(p + ".conv3", width * 4, width, 1)
            bn(p + ".bn3", width * 4)
            if b == 0:
                conv(p + ".downsample.0", width * 4, cin, 1)
                bn(p + ".downsample.1", width * 4)
            cin = width * 4
    out.append(("fc.weight", (1000 // d) * (2048 // d)))
    out.append(("fc.bias", 1000 // d))
    return out


def lstm_lm_shapes(hidden: int = 1500, vocab: int = 10_000, layers: int = 2) -> list[tuple[str, int]]:
    """Embedding, ``layers`` LSTM layers (4 gates) and the decoder of a word LM."""
    out = [("embedding.weight", vocab * hidden)]
    for l in range(layers):
        out += [(f"lstm.weight_ih_l{l}", 4 * hidden * hidden),
                (f"lstm.weight_hh_l{l}", 4 * hidden * hidden),
                (f"lstm.bias_ih_l{l}", 4 * hidden),
                (f"lstm.bias_hh_l{l}", 4 * hidden)]
    out += [("decoder.weight", vocab * hidden), ("decoder.bias", vocab)]
    return out


def vgg16_conv_shapes(width_div: int = 1) -> list[tuple[str, int]]:
    """The 13 3x3 convolutions (+ biases) of VGG-16's feature stack."""
    plan = [64, 64, 128, 128, 256, 256, 256, 512, 512, 512, 512, 512, 512]
    out, cin = [], 3
    for i, c in enumerate(plan):
        c //= width_div
        out.append((f"features.{i}.weight", c * cin * 9))
        out.append((f"features.{i}.bias", c))
        cin = c
    return out


def deepspeech_shapes(rows: int = 2560, cols: int = 7680, n_big: int = 5, n_out: int = 29) -> list[tuple[str, int]]:
    """GRU-sized recurrent weight tensors plus the character output layer."""
    return [(f"rnn.{i}.weight", rows * cols) for i in range(n_big)] + [("fc.weight", rows * n_out)]


# --------------------------------------------------------------------------
# configurations
# --------------------------------------------------------------------------

@dataclass
class Workload:
    """One synthetic workload: a flat layout of segments and its knobs."""
    config: int
    name: str
    sizes: list[int]
    learners: int
    steps: int
    method: str                      # "dgc", "adacomp" or "dcd"
    density: float = 0.001
    momentum: float = 0.9
    clip_thr: float = 0.0
    clip_nodes: int = 1
    lt: list[int] = field(default_factory=list)   # AdaComp bin length per segment
    also_adacomp_lt: int = 0         # config 1 runs AdaComp on the same tensor too
    gamma: float = 0.1               # DCD step size
    keep_p: float = 0.01             # DCD random-sparsification keep probability
    ring_w: tuple = (1.0 / 3.0, 1.0 / 3.0, 1.0 / 3.0)

    @property
    def n(self) -> int:
        return int(sum(self.sizes))

    @property
    def offsets(self) -> np.ndarray:
        return layout_offsets(self.sizes)


def layout_offsets(sizes) -> np.ndarray:
    off = np.zeros(len(sizes) + 1, dtype=np.int64)
    np.cumsum(np.asarray(sizes, dtype=np.int64), out=off[1:])
    return off


def workload(config: int, small: bool = False) -> Workload:
    """The five configurations; ``small`` shrinks them for oracle-speed tests."""
    if config == 1:
        n = 1_048_576 if not small else 65_536
        return Workload(1, "dgc_single_1M" if not small else "dgc_single_64k", [n], learners=1, steps=3,
                        method="dgc", clip_thr=1.0, clip_nodes=1, also_adacomp_lt=50)
    if config == 2:
        shapes = resnet50_shapes(1 if not small else 8)
        return Workload(2, "resnet50_dgc_k4" if not small else "resnet50_div8_dgc_k4",
                        [s for _, s in shapes], learners=4, steps=5, method="dgc")
    if config == 3:
        lstm = lstm_lm_shapes() if not small else lstm_lm_shapes(hidden=150, vocab=1000)
        vgg = vgg16_conv_shapes(1 if not small else 8)
        sizes = [s for _, s in lstm] + [s for _, s in vgg]
        lt = [500] * len(lstm) + [50] * len(vgg)
        return Workload(3, "lstm_vgg_adacomp_k8" if not small else "lstm150_vgg_div8_adacomp_k8",
                        sizes, learners=8, steps=5, method="adacomp", lt=lt)
    if config == 4:
        shapes = deepspeech_shapes() if not small else deepspeech_shapes(256, 768)
        return Workload(4, "deepspeech_dgc_k8" if not small else "deepspeech_small_dgc_k8",
                        [s for _, s in shapes], learners=8, steps=10, method="dgc")
    if config == 5:
        d = 25_600_000 if not small else 262_144
        return Workload(5, "dcd_ring8" if not small else "dcd_ring8_small", [d], learners=8, steps=10,
                        method="dcd")
    raise ValueError(f"unknown config {config}")


# --------------------------------------------------------------------------
# seeded draws
# --------------------------------------------------------------------------

def seed_for(config: int, learner: int, step: int) -> int:
    return 1000 * config + 100 * learner + step


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def per_tensor_log_uniform(config: int, count: int, lo_exp: float, hi_exp: float) -> np.ndarray:
    """One scale per tensor, 10**U(lo_exp, hi_exp), fixed for the configuration."""
    g = _gen(1000 * config + 999, "cpu")
    u = torch.rand(count, generator=g, dtype=torch.float64)
    return (10.0 ** (lo_exp + (hi_exp - lo_exp) * u)).numpy()


def _expand(scales: np.ndarray, sizes, device) -> torch.Tensor:
    return torch.repeat_interleave(torch.as_tensor(scales, dtype=torch.float32),
                                   torch.as_tensor(np.asarray(sizes, dtype=np.int64))).to(device)


def gradient(w: Workload, learner: int, step: int, device="cpu") -> torch.Tensor:
    """The synthetic fp32 gradient (DGC) or new gradient dW (AdaComp) of one learner at one step."""
    g = _gen(seed_for(w.config, learner, step), device)
    n = w.n
    if w.config == 1:
        return torch.randn(n, generator=g, device=device, dtype=torch.float32) * 1e-3
    if w.config == 2:
        sig = _expand(per_tensor_log_uniform(2, len(w.sizes), -5.0, -2.0), w.sizes, device)
        return torch.randn(n, generator=g, device=device, dtype=torch.float32) * sig
    if w.config == 3:
        b = _expand(per_tensor_log_uniform(3, len(w.sizes), -6.0, -3.0), w.sizes, device)
        # Laplace(0, b) by inversion of its CDF
        u = torch.rand(n, generator=g, device=device, dtype=torch.float32) - 0.5
        u = u.clamp(-0.4999999, 0.4999999)
        return (-b * torch.sign(u) * torch.log1p(-2.0 * u.abs())).to(torch.float32)
    if w.config == 4:
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32) * 1e-4
        heavy = torch.rand(n, generator=g, device=device, dtype=torch.float32) < 0.01
        return torch.where(heavy, x * 100.0, x)
    if w.config == 5:
        return torch.randn(n, generator=g, device=device, dtype=torch.float32) * 1e-3
    raise ValueError(w.config)


def gradients(w: Workload, step: int, device="cpu") -> torch.Tensor:
    """[K, N] stack of every learner's gradient at ``step``."""
    return torch.stack([gradient(w, k, step, device) for k in range(w.learners)])


def dcd_initial_model(w: Workload, device="cpu") -> torch.Tensor:
    """x_0 ~ N(0, 1e-2^2), one vector shared by all nodes, as [n_nodes, D]."""
    g = _gen(1000 * w.config + 999, device)
    x0 = torch.randn(w.n, generator=g, device=device, dtype=torch.float32) * 1e-2
    return x0.unsqueeze(0).repeat(w.learners, 1)


def dcd_seed(w: Workload) -> int:
    """Key of the counter-based generator that draws the sparsification masks."""
    return 0x5EED_0000_0000_0000 + w.config


def random_layout(rng: np.random.Generator, n_seg: int, max_len: int, min_len: int = 0) -> list[int]:
    """Ragged segment sizes for edge-case tests (may contain empty segments)."""
    return [int(x) for x in rng.integers(min_len, max_len + 1, size=n_seg)]


def human_bytes(b: float) -> str:
    for unit in ("B", "KB", "MB", "GB", "TB"):
        if abs(b) < 1000 or unit == "TB":
            return f"{b:.1f} {unit}"
        b /= 1000.0
    return f"{b:.1f} TB"


__all__ = [name for name in dir() if not name.startswith("_") and name not in ("annotations", "math")]
