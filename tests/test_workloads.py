"""The synthetic workloads against the numbers the pages print (tests/golden)."""
import json
import os

import numpy as np
import pytest
import torch

from checkpoint_averaging_gb300 import workloads as W

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def fact(key):
    return GOLD[key]["value"]


def rounds_to(x, key):
    g = GOLD[key]
    return abs(x - g["value"]) <= g["rounding"] / 2 + 1e-12


def test_pythia14m_shapes_match_page():
    wl = W.workload("pythia14m")
    names = [s.name for s in wl.specs]
    layers = {n.split(".")[2] for n in names if ".layers." in n}
    assert len(layers) == fact("pythia14m_layers")
    assert wl.specs[0].shape[1] == fact("pythia14m_width")
    assert rounds_to(wl.n_params / 1e6, "pythia14m_params_millions")
    emb = sum(s.numel for s in wl.specs if "embed" in s.name)
    assert rounds_to(emb / 1e6, "pythia14m_embedding_params_millions")
    for f in (0, 3):  # each embedding is its own fp32 fragment
        assert rounds_to(wl.fragment_numel(f) * 4 / 1e6, "pythia14m_embedding_fragment_mb_fp32")
    assert wl.n_fragments == fact("gradientmail_fragments")
    assert wl.quorum == fact("gradientmail_quorum")
    assert wl.lr == fact("gradientmail_outer_lr") and wl.mu == fact("gradientmail_outer_momentum")
    # the blocks occupy the other two fragments
    assert {s.fragment for s in wl.specs if ".layers." in s.name} == {1, 2}


def test_diffurefill1b_shapes_match_page():
    for wl in (W.workload("diffurefill1b"), W.workload("diffurefill1b_bf16")):
        assert rounds_to(wl.n_params / 1e9, "diffurefill_params_billions")
        emb = wl.specs[0]
        assert emb.shape == (fact("diffurefill_vocab"), fact("diffurefill_width"))
        blocks = {s.name.split(".")[1] for s in wl.specs if s.name.startswith("blocks.")}
        assert len(blocks) == fact("diffurefill_layers")
        assert any(s.shape == (fact("diffurefill_ffn"), fact("diffurefill_width")) for s in wl.specs)
        # tied embedding: no separate output head
        assert sum(1 for s in wl.specs if s.shape[0] == fact("diffurefill_vocab")) == 1
    assert W.workload("diffurefill1b").ema_beta == fact("diffurefill_ema_beta")
    assert W.workload("diffurefill1b").lr == fact("diffurefill_replacement_outer_lr")


def test_fragment_sizes_1b():
    wl = W.workload("diffurefill1b_bf16")
    assert [wl.fragment_numel(f) for f in range(4)] == [151_060_480, 308_305_920,
                                                         308_305_920, 308_307_968]
    assert wl.fragment_numel(-1) == 1_075_980_288


def test_sweep_lists_are_ragged_and_sum_to_total():
    for t, n in W.SWEEP_POINTS:
        specs = W.sweep_specs(t, n)
        sizes = np.array([s.numel for s in specs])
        assert len(specs) == t and sizes.sum() == n
        assert not (sizes % 8 == 0).any()
        assert sizes.max() <= 150_000_000


def test_round_draws_are_seeded_and_respect_quorum():
    wl = W.workload("diffurefill1b_bf16")
    a, b = W.draw_round(wl, 0, 0), W.draw_round(wl, 0, 0)
    assert a == b
    assert len(a.included) == wl.K - wl.n_masked >= wl.quorum
    assert all(100_000 <= t <= 150_000 for t in a.tokens)
    assert W.draw_round(wl, 1, 0) != a


def test_generated_inputs_are_aligned_and_seeded():
    wl = W.workload("pythia14m")
    g1 = W.make_global(wl, 0, "cpu")
    g2 = W.make_global(wl, 0, "cpu")
    assert torch.equal(g1.flat, g2.flat)
    for v in g1.views:
        assert v.data_ptr() % 256 == 0
    w = W.make_worker(wl, g1, 0, 1, 0, "cpu")
    d = (w.flat - g1.flat)
    assert 0.5e-3 < d.std().item() < 2e-3
    assert 0.015 < g1.flat[:g1.numels[0]].std().item() < 0.025


def test_bf16_workers_are_rounded_fp32_workers():
    wl = W.workload("diffurefill1b_bf16")
    small = W.Workload("tiny", tuple(W.sweep_specs(4, 40_000)), 1, K=2, n_masked=0,
                       quorum=2, ckpt_dtype="bf16", mode="delta")
    g = W.make_global(small, 0, "cpu")
    w = W.make_worker(small, g, 0, 0, 0, "cpu")
    assert w.flat.dtype == torch.bfloat16
    assert wl.ckpt_dtype == "bf16"


def test_workload_name_modifiers():
    base = W.workload("stand")
    swa = W.workload("stand+swa")
    assert swa.swa and not base.swa and swa.specs == base.specs
    wn = W.workload("sweep:64,16000000,3,wnorms-ema")
    assert wn.ema_beta is None and wn.norms and wn.worker_norms
    assert W.workload("sweep:64,16000000,3").ema_beta == 0.9
