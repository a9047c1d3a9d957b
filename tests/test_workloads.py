"""The seeded input recipe (muonh_workloads.py) against what it states: the
shapes and parameter counts of every workload, seeding that makes any subset
equal the same matrices of a full draw, and the distributions of weights and
gradients (normal, Student-t with 3 degrees of freedom, rank 8 plus noise)."""

import numpy as np
import pytest
import torch

import muonh_workloads as wl


def test_shapes_and_parameter_counts():
    full = wl.qwen3_2b()
    assert len(full.shapes) == 196 and full.n_params == 1_409_286_144
    layer = wl.qwen3_layer()
    assert layer.shapes == [(2048, 2048), (1024, 2048), (1024, 2048), (2048, 2048), (6144, 2048), (6144, 2048),
                            (2048, 6144)]
    assert full.shapes == layer.shapes * 28
    assert wl.qwen3_2b(layers=4).shapes == layer.shapes * 4
    b = wl.batched_256()
    assert b.shapes == [(256, 256)] * 1024 and b.grad_kind == "student_t3"
    a = wl.aspect_16384x1024()
    assert a.shapes == [(16384, 1024)] * 4 + [(1024, 16384)] * 4 and a.grad_kind == "low_rank8"
    ad = wl.adamw_group()
    assert ad.shapes[0] == (151936, 2048) and len(ad.shapes) == 1 + 57 + 56
    assert wl.single_256x128().shapes == [(256, 128)]
    assert set(wl.ALL) == {"single_256x128", "qwen3_layer_d2048", "qwen3_2b_28layers", "batched_1024x256x256",
                           "aspect_16384x1024", "qwen3_2b_adamw_group"}


def test_seeding_is_per_matrix_and_per_step():
    work = wl.ragged([(16, 8), (8, 16), (16, 8)])
    w_all = work.weights()
    assert torch.equal(work.weights(indices=[2])[0], w_all[2])        # a subset equals the full draw
    assert not torch.equal(w_all[0], w_all[2])                        # same shape, different matrix
    assert torch.equal(work.grads(3)[1], work.grad(1, 3))
    assert not torch.equal(work.grad(1, 3), work.grad(1, 4))          # a fresh gradient every step
    assert torch.equal(wl.ragged([(16, 8)]).weight(0), w_all[0])     # seeds depend on the index only


def test_weight_and_normal_gradient_scales():
    work = wl.ragged([(512, 512)])
    w = work.weight(0).double().numpy()
    g = work.grad(0, 0).double().numpy()
    assert abs(w.std() / 0.02 - 1) < 0.01 and abs(w.mean()) < 0.02 * 0.01
    assert abs(g.std() / 1e-3 - 1) < 0.01


def test_student_t3_gradients():
    # median |t_3| = 0.7649 (Student-t with 3 degrees of freedom); heavy tails:
    # P(|t_3| > 5) = 0.0154, against 5.7e-7 for a normal
    g = wl.ragged([(512, 512)], grad_kind="student_t3").grad(0, 0).double().numpy() / 1e-3
    a = np.abs(g)
    assert abs(np.median(a) / 0.7649 - 1) < 0.02
    assert abs((a > 5).mean() / 0.0154 - 1) < 0.1


def test_low_rank8_gradients():
    g = wl.ragged([(300, 200)], grad_kind="low_rank8").grad(0, 0).double().numpy()
    s = np.linalg.svd(g, compute_uv=False)
    assert s[7] > 1e3 * s[8]                                          # rank 8 plus 1e-5 noise
    assert s[8] < 1e-5 * 3 * np.sqrt(300)
