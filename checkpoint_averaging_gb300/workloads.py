"""Seeded synthetic merge workloads shaped like the models on the pages.

This module holds no merge arithmetic. It lists parameter shapes, assigns
tensors to fragments, and draws seeded inputs: the starting global, the
workers' checkpoints, their token counts and which workers make the quorum.
The CUDA path and the CPU oracle are fed the very same arrays from here.

Shapes come from:
  * "Pythia-14M on four rented GPUs and a bucket", "Choosing a reference run":
    six layers of width 128, 14 million parameters, 12.9 million of them in its
    two embeddings; "Getting updates through the bucket": fragments=4, each
    embedding a 25.8 MB fp32 fragment, the transformer blocks the other two.
  * "DiffuRefill-1B: Pretraining a Masked Diffusion Language Model on Free,
    Preemptible Notebook GPUs", section 2, Table 1: 1.08B parameters, embedding
    tied to the output head, 18 layers of width 2048, SwiGLU 5632, RMSNorm,
    vocabulary 73,760.
  * "DiffuRefill-1B" model card, "What the run taught": the 37.9M-parameter
    stand (8 blocks, width 512, SwiGLU 1408, tied 73,760 x 512 embedding).

Value distributions follow the workload descriptions: global ~ N(0, 0.02),
worker = global + N(0, sigma) per round, token counts uniform integers,
bf16 checkpoints are the fp32 worker values rounded to nearest-even.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

# Every tensor view starts on a multiple of this many elements inside its
# arena (512 B for fp32, 256 B for bf16), so 16- and 32-byte vector loads
# are legal on every tensor of a generated workload.
ALIGN_ELEMS = 128

_MASK64 = (1 << 64) - 1


def _splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def subseed(*keys) -> int:
    """A 63-bit seed derived from an ordered tuple of ints/strings."""
    h = 0x0123456789ABCDEF
    for k in keys:
        if isinstance(k, str):
            for b in k.encode():
                h = _splitmix64(h ^ b)
        else:
            h = _splitmix64(h ^ (int(k) & _MASK64))
    return h & ((1 << 63) - 1)


@dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple
    fragment: int = 0

    @property
    def numel(self) -> int:
        return int(math.prod(self.shape))


# ---- parameter lists --------------------------------------------------------

def pythia14m_specs() -> list[TensorSpec]:
    """GPT-NeoX Pythia-14M: embed_in, 6 layers of width 128 (4x MLP), final
    LayerNorm, untied embed_out. Fragments: {embed_in}, {layers 0-2},
    {layers 3-5 + final norm}, {embed_out}."""
    V, d = 50304, 128
    specs = [TensorSpec("gpt_neox.embed_in.weight", (V, d), 0)]
    for i in range(6):
        f = 1 if i < 3 else 2
        p = f"gpt_neox.layers.{i}."
        specs += [
            TensorSpec(p + "input_layernorm.weight", (d,), f),
            TensorSpec(p + "input_layernorm.bias", (d,), f),
            TensorSpec(p + "post_attention_layernorm.weight", (d,), f),
            TensorSpec(p + "post_attention_layernorm.bias", (d,), f),
            TensorSpec(p + "attention.query_key_value.weight", (3 * d, d), f),
            TensorSpec(p + "attention.query_key_value.bias", (3 * d,), f),
            TensorSpec(p + "attention.dense.weight", (d, d), f),
            TensorSpec(p + "attention.dense.bias", (d,), f),
            TensorSpec(p + "mlp.dense_h_to_4h.weight", (4 * d, d), f),
            TensorSpec(p + "mlp.dense_h_to_4h.bias", (4 * d,), f),
            TensorSpec(p + "mlp.dense_4h_to_h.weight", (d, 4 * d), f),
            TensorSpec(p + "mlp.dense_4h_to_h.bias", (d,), f),
        ]
    specs += [TensorSpec("gpt_neox.final_layer_norm.weight", (d,), 2),
              TensorSpec("gpt_neox.final_layer_norm.bias", (d,), 2),
              TensorSpec("embed_out.weight", (V, d), 3)]
    return specs


def _llama_like_specs(vocab: int, dim: int, ffn: int, blocks: int,
                      fragments: int) -> list[TensorSpec]:
    """Tied embedding, `blocks` pre-norm blocks (q, k, v, o, SwiGLU gate/up/
    down, two RMSNorm weights), final norm. With fragments == 4 the split is
    {embedding}, then the blocks in three equal runs, the final norm joining
    the last run."""
    def frag_of_block(i: int) -> int:
        if fragments == 1:
            return 0
        per = blocks // (fragments - 1)
        return min(1 + i // per, fragments - 1)

    specs = [TensorSpec("embed.weight", (vocab, dim), 0)]
    for i in range(blocks):
        f = frag_of_block(i)
        p = f"blocks.{i}."
        specs += [
            TensorSpec(p + "attn.q.weight", (dim, dim), f),
            TensorSpec(p + "attn.k.weight", (dim, dim), f),
            TensorSpec(p + "attn.v.weight", (dim, dim), f),
            TensorSpec(p + "attn.o.weight", (dim, dim), f),
            TensorSpec(p + "mlp.gate.weight", (ffn, dim), f),
            TensorSpec(p + "mlp.up.weight", (ffn, dim), f),
            TensorSpec(p + "mlp.down.weight", (dim, ffn), f),
            TensorSpec(p + "norm1.weight", (dim,), f),
            TensorSpec(p + "norm2.weight", (dim,), f),
        ]
    specs.append(TensorSpec("final_norm.weight", (dim,), fragments - 1))
    return specs


def stand_specs() -> list[TensorSpec]:
    """The stand: 8 blocks, width 512, SwiGLU 1408, tied 73,760 x 512."""
    return _llama_like_specs(73760, 512, 1408, 8, fragments=1)


def diffurefill1b_specs(fragments: int = 1) -> list[TensorSpec]:
    """DiffuRefill-1B: 18 blocks, width 2048, SwiGLU 5632, tied 73,760 x 2048."""
    return _llama_like_specs(73760, 2048, 5632, 18, fragments=fragments)


def sweep_specs(n_tensors: int, total: int, seed: int = 0) -> list[TensorSpec]:
    """Ragged list of n_tensors 1-D tensors summing to `total` elements: sizes
    log-uniform over [2048, 150e6], rescaled to the total, clamped, the
    remainder given to the largest; sizes that are multiples of 8 are nudged
    by one so that every tensor has a ragged tail."""
    lo, hi = 2048, 150_000_000
    rng = np.random.default_rng(subseed(seed, "sweep", n_tensors, total))
    raw = np.exp(rng.uniform(math.log(lo), math.log(hi), n_tensors))
    sizes = np.clip(np.floor(raw * (total / raw.sum())), lo, hi).astype(np.int64)
    big = int(np.argmax(sizes))
    sizes[big] += total - int(sizes.sum())
    for i in range(n_tensors):
        if i != big and sizes[i] % 8 == 0:
            sizes[i] += 1
            sizes[big] -= 1
    if sizes[big] % 8 == 0:
        j = next(i for i in range(n_tensors) if i != big and sizes[i] % 8 not in (0, 7))
        sizes[big] -= 1
        sizes[j] += 1
    assert int(sizes.sum()) == total and (sizes > 0).all()
    assert n_tensors == 1 or not (sizes % 8 == 0).any()
    return [TensorSpec(f"sweep.{i}", (int(s),), 0) for i, s in enumerate(sizes)]


# ---- workloads --------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    specs: tuple
    n_fragments: int
    K: int                      # workers that push a checkpoint each round
    n_masked: int               # of those, how many miss the round
    quorum: int
    ckpt_dtype: str             # "f32" or "bf16"
    mode: str                   # "mean" (plain replacement) or "delta" (Nesterov)
    lr: float = 1.0
    mu: float = 0.0
    ema_beta: float | None = None
    rounds: tuple = ((0, -1),)  # (round number, fragment or -1 for all)
    in_flight: int = 1          # rounds committed together on separate streams
    global_std: float = 0.02
    noise_std: float = 1e-3
    tokens: tuple | None = None  # inclusive integer range
    norms: bool = False
    workers_track_global: bool = False  # workers start from the current global
    swa: bool = False                   # also fold each global into the uniform average
    worker_norms: bool = False          # also report each worker's own drift
    share_sms: bool = False             # merge passes leave room for rounds in flight beside them
    commit_many: int = 0                # rounds committed together by one call (0: one per call)

    @property
    def n_params(self) -> int:
        return sum(s.numel for s in self.specs)

    @property
    def fragment_of(self) -> list[int]:
        return [s.fragment for s in self.specs]

    def fragment_numel(self, fragment: int) -> int:
        return sum(s.numel for s in self.specs if fragment == -1 or s.fragment == fragment)


def _wl_pythia() -> Workload:
    # three fragment rounds per step; as in the Pythia page's run ("Getting
    # updates through the bucket"), two rounds may be in flight at once, and
    # their merge passes share the SMs (the long round beside the short ones)
    return Workload("pythia14m_f4_q3_delta_nesterov", tuple(pythia14m_specs()), 4,
                    K=4, n_masked=1, quorum=3, ckpt_dtype="f32", mode="delta",
                    lr=0.7, mu=0.9, rounds=((0, 0), (1, 1), (2, 2)), in_flight=2,
                    noise_std=1e-3, tokens=(200_000, 600_000), norms=True, share_sms=True)


def _wl_stand() -> Workload:
    return Workload("stand63m_k5_mean_ema", tuple(stand_specs()), 1, K=5, n_masked=0,
                    quorum=5, ckpt_dtype="f32", mode="mean", ema_beta=0.9,
                    rounds=tuple((r, -1) for r in range(10)), noise_std=2e-3,
                    workers_track_global=True)


def _wl_1b() -> Workload:
    return Workload("diffurefill1b_k5_f32_mean_ema", tuple(diffurefill1b_specs(1)), 1,
                    K=5, n_masked=0, quorum=5, ckpt_dtype="f32", mode="mean",
                    ema_beta=0.9, rounds=((0, -1),), noise_std=1e-3)


def _wl_1b_swa() -> Workload:
    """The 1.08B round of the final stretch: plain mean + EMA + the uniform
    average of the globals, all in one pass."""
    return Workload("diffurefill1b_k5_f32_mean_ema_swa", tuple(diffurefill1b_specs(1)), 1,
                    K=5, n_masked=0, quorum=5, ckpt_dtype="f32", mode="mean",
                    ema_beta=0.9, rounds=((0, -1),), noise_std=1e-3, swa=True)


def _wl_1b_bf16_wnorms() -> Workload:
    """The bf16 fragment rounds with each worker's own drift reported too."""
    w = _wl_1b_bf16()
    return Workload(w.name + "_wnorms", w.specs, w.n_fragments, K=w.K, n_masked=w.n_masked,
                    quorum=w.quorum, ckpt_dtype=w.ckpt_dtype, mode=w.mode, lr=w.lr, mu=w.mu,
                    rounds=w.rounds, in_flight=w.in_flight, noise_std=w.noise_std,
                    tokens=w.tokens, norms=True, worker_norms=True)


def _wl_1b_bf16() -> Workload:
    return Workload("diffurefill1b_bf16_f4_q3_delta_nesterov_norms",
                    tuple(diffurefill1b_specs(4)), 4, K=5, n_masked=2, quorum=3,
                    ckpt_dtype="bf16", mode="delta", lr=0.7, mu=0.9,
                    rounds=((0, 0), (1, 1)), in_flight=2, noise_std=1e-3,
                    tokens=(100_000, 150_000), norms=True)


def sweep_workload(n_tensors: int, total: int, K: int, seed: int = 0) -> Workload:
    return Workload(f"sweep_t{n_tensors}_n{total}_k{K}_bf16",
                    tuple(sweep_specs(n_tensors, total, seed)), 1, K=K, n_masked=0,
                    quorum=K, ckpt_dtype="bf16", mode="delta", lr=0.7, mu=0.9,
                    ema_beta=0.9, rounds=((0, -1),), noise_std=1e-3,
                    tokens=(100_000, 150_000))


SWEEP_POINTS = ((64, 16_000_000), (128, 256_000_000), (256, 1_000_000_000),
                (512, 4_000_000_000))
SWEEP_K = (2, 4, 8)


def workload(name: str) -> Workload:
    """A workload by name; a "+swa" suffix also folds each global into the
    uniform running average, a "-ema" suffix drops the EMA update, a "+wnorms"
    suffix asks for the round's and each worker's drift norms."""
    import dataclasses
    if name.endswith("+wnorms"):
        wl = workload(name[:-len("+wnorms")])
        return dataclasses.replace(wl, name=wl.name + "_wnorms", norms=True, worker_norms=True)
    if name.endswith("+swa"):
        wl = workload(name[:-len("+swa")])
        return dataclasses.replace(wl, name=wl.name + "_swa", swa=True)
    if name.endswith("-ema"):
        wl = workload(name[:-len("-ema")])
        return dataclasses.replace(wl, name=wl.name + "_noema", ema_beta=None)
    table = {
        "pythia14m": _wl_pythia,
        "stand": _wl_stand,
        "diffurefill1b": _wl_1b,
        "diffurefill1b_bf16": _wl_1b_bf16,
        "diffurefill1b_swa": _wl_1b_swa,
        "diffurefill1b_bf16_wnorms": _wl_1b_bf16_wnorms,
    }
    if name in table:
        return table[name]()
    if name.startswith("sweep:"):
        parts = name.split(":")[1].split(",")
        t, n, k = (int(v) for v in parts[:3])
        wl = sweep_workload(t, n, k)
        if len(parts) > 3 and parts[3] == "norms":  # Nesterov + EMA + drift norms
            wl = dataclasses.replace(wl, name=wl.name + "_norms", norms=True)
        elif len(parts) > 3 and parts[3] == "wnorms":  # ... plus each worker's drift
            wl = dataclasses.replace(wl, name=wl.name + "_wnorms", norms=True, worker_norms=True)
        return wl
    raise KeyError(name)


# ---- seeded draws -----------------------------------------------------------

@dataclass
class Arena:
    """One flat buffer holding a whole tensor list, each tensor at an offset
    that is a multiple of ALIGN_ELEMS elements."""
    flat: torch.Tensor
    offsets: list
    numels: list
    views: list = field(default_factory=list)

    def __post_init__(self):
        self.views = [self.flat[o:o + n] for o, n in zip(self.offsets, self.numels)]


def arena_layout(numels) -> tuple[list, int]:
    offs, pos = [], 0
    for n in numels:
        offs.append(pos)
        pos += -(-max(int(n), 1) // ALIGN_ELEMS) * ALIGN_ELEMS
    return offs, pos


def empty_arena(numels, dtype, device) -> Arena:
    """Zeroed arena whose base (and so every tensor view) is 512-byte aligned."""
    offs, total = arena_layout(numels)
    esize = torch.empty(0, dtype=dtype).element_size()
    slack = 512 // esize
    raw = torch.zeros(total + slack, dtype=dtype, device=device)
    skip = (-raw.data_ptr() % 512) // esize
    return Arena(raw[skip:skip + total], offs, [int(n) for n in numels])


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


_CHUNK = 1 << 28  # draw at most 256M values per call to bound temporaries


def _normal_(flat: torch.Tensor, std: float, gen: torch.Generator) -> None:
    for s in range(0, flat.numel(), _CHUNK):
        flat[s:s + _CHUNK].normal_(0.0, std, generator=gen)


def make_global(wl: Workload, seed: int, device) -> Arena:
    """The starting global: fp32 ~ N(0, global_std)."""
    a = empty_arena([s.numel for s in wl.specs], torch.float32, device)
    _normal_(a.flat, wl.global_std, _gen(subseed(seed, wl.name, "global"), device))
    return a


def make_worker(wl: Workload, base: Arena, round: int, worker: int, seed: int,
                device, out: Arena | None = None) -> Arena:
    """Worker `worker`'s checkpoint for `round`: base + N(0, noise_std), stored
    as the workload's checkpoint dtype (bf16 rounded to nearest-even)."""
    dt = torch.bfloat16 if wl.ckpt_dtype == "bf16" else torch.float32
    if out is None:
        out = empty_arena(base.numels, dt, device)
    gen = _gen(subseed(seed, wl.name, "worker", round, worker), device)
    n = base.flat.numel()
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        tmp = torch.empty(e - s, dtype=torch.float32, device=device)
        tmp.normal_(0.0, wl.noise_std, generator=gen)
        tmp.add_(base.flat[s:e].to(device))
        out.flat[s:e].copy_(tmp)  # fp32 -> bf16 copy rounds to nearest-even
        del tmp
    return out


@dataclass
class RoundDraw:
    round: int
    fragment: int
    tokens: list          # per worker (all K), ints
    included: list        # workers that made the round, in arrival order


def draw_round(wl: Workload, index: int, seed: int) -> RoundDraw:
    """Token counts, the masked workers and the arrival order for round index
    `index` of the workload."""
    rnd, frag = wl.rounds[index]
    g = torch.Generator().manual_seed(subseed(seed, wl.name, "round", rnd))
    if wl.tokens is not None:
        lo, hi = wl.tokens
        tokens = torch.randint(lo, hi + 1, (wl.K,), generator=g).tolist()
    else:
        tokens = [0] * wl.K
    order = torch.randperm(wl.K, generator=g).tolist()
    masked = set(order[:wl.n_masked])
    arrival = torch.randperm(wl.K, generator=g).tolist()
    included = [k for k in arrival if k not in masked]
    return RoundDraw(rnd, frag, [int(t) for t in tokens], included)
