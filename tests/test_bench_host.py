"""Host logic of bench.py that needs no GPU: the multi-rank timing reduction
(two gloo ranks on CPU), whole-job rates, launch counting, algorithmic bytes
and the reference arm's rank handling."""
import io
import os
import socket
import sys
import contextlib

import pytest

import bench
from trellis_decode_gemv_gb300 import synth


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp

    from tests import dist_helpers

    world = 2
    mp.spawn(dist_helpers.max_over_ranks_worker, args=(world, _free_port(), str(tmp_path)),
             nprocs=world, join=True)
    vals = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    for t, rate in vals:
        assert float(t) == 2.5  # the slowest rank's time on every rank
        assert float(rate) == pytest.approx(1000.0 * 2 * 10 / 2.5)


def test_single_process_reduction_is_identity():
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    bench.barrier()  # no process group: a no-op
    assert bench.whole_job_rate(5.0, 1, 4, 2.0) == 10.0


def test_kernels_per_call():
    sms = 152
    # decode-MMA kernel (M > 2, or forced): one launch at batch 1 and 2, plus the operand-image kernel above
    assert bench.kernels_per_call("tensor", 1, 4096, 4096, sms) == 1
    assert bench.kernels_per_call("tensor", 2, 14336, 4096, sms) == 1
    assert bench.kernels_per_call("auto", 3, 4096, 4096, sms) == 2
    assert bench.kernels_per_call("auto", 32, 4096, 4096, sms) == 2
    # warp-shuffle (AUTO at batch <= 2), small layer at batch 1: segment kernel + output kernel
    assert bench.kernels_per_call("auto", 1, 4096, 4096, sms) == 2
    assert bench.kernels_per_call("shuffle", 1, 4096, 4096, sms) == 2
    # large layer at batch 1: x pairs + sub-unit kernel + output kernel
    assert bench.kernels_per_call("auto", 1, 14336, 4096, sms) == 3
    # forced warp-shuffle batch 5 on a small layer: chunk of 4 (3 kernels) + chunk of 1 (2)
    assert bench.kernels_per_call("shuffle", 5, 1024, 4096, sms) == 5


def test_algorithmic_bytes_and_ops():
    w, b, ops = bench.algorithmic(4096, 4096, 2, synth.CB_1MAD, 1)
    assert w == 4096 * 4096
    assert b == 4096 * 4096 * 2 // 8 + 2 * 4096 + 2 * (4096 + 4096) + 2 * 4096 + 2 * 4096
    assert ops == w * 5
    assert bench.algorithmic(128, 256, 3, synth.CB_3INST, 2)[2] == 128 * 256 * 4


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(workload="single", batch=1, steps=1, warmup=0, gpus=2)
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert bench.run_reference(args) == 0
    assert out.getvalue() == ""


def test_decoder_groups():
    g = bench.decoder_groups(synth.llama8b_layer_set())
    assert len(g) == 24  # per (K, code): [q, k, v], [o], [gate, up], [down]
    assert g[:4] == [[0, 1, 2], [3], [4, 5], [6]]
    assert sum(len(x) for x in g) == 42
    assert all(len(x) == 1 for x in bench.decoder_groups(synth.llama8b_layer_set(), grouped=False))
    # gate and up of the mixed stack are grouped only when their widths agree
    gemvs = synth.mixed_stack()
    for x in bench.decoder_groups(gemvs):
        assert len({(gemvs[i][3], gemvs[i][4]) for i in x}) == 1


def test_kernels_per_group():
    sms = 152
    # warp-shuffle at batch <= 2: x pairs, one sub-unit kernel over every layer, output transform
    assert bench.kernels_per_group("auto", 1, [(4096, 4096), (1024, 4096), (1024, 4096)], sms) == 3
    # decode-MMA above: one image launch for every layer, one launch over every layer
    assert bench.kernels_per_group("auto", 5, [(4096, 4096), (1024, 4096)], sms) == 2
    assert bench.kernels_per_group("tensor", 1, [(4096, 4096), (1024, 4096)], sms) == 1
    assert bench.kernels_per_group("shuffle", 5, [(4096, 4096), (1024, 4096)], sms) == 6
    assert bench.kernels_per_group("auto", 1, [(1024, 4096)], sms) == 2


def test_launches_of_multi_code_groups():
    """A multi-code call: one input and one output kernel around a layer
    kernel per (K, code) class and batch chunk (int8: chunks of 8/4/2/1 rows)."""
    sms, shapes = 152, [(4096, 4096), (1024, 4096), (1024, 4096)]
    kcs = [(2, 1), (3, 3), (2, 1)]
    assert bench.launches_of_group(None, "auto", 1, shapes, sms, False, True, kcs) == 4
    assert bench.launches_of_group(None, "auto", 3, shapes, sms, False, True, kcs) == 6
    assert bench.launches_of_group(None, "auto", 1, shapes, sms, False, True) == 3
    assert bench.launches_of_group(None, "auto", 2, shapes, sms, False, False, kcs) == 4
    # batch 1, the llama8b step: K = 2, 3, 4 each with 3INST and 1MAD, 218 M
    # weights per class: one launch per K between the x-pair and output kernels
    step = [(m, n) for m, n in [(4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096), (14336, 4096),
                                (14336, 4096), (4096, 14336)]]
    shs, kc6 = [], []
    for K in (2, 3, 4):
        for cb in (0, 1):
            shs += step
            kc6 += [(K, cb)] * len(step)
    assert bench.launches_of_group(None, "auto", 1, shs, sms, False, False, kc6) == 5
    # the int8 path the same way (1MAD and mul1 of one K share a launch)
    kc6b = [(K, 1 if cb == 0 else 3) for K, cb in kc6]
    assert bench.launches_of_group(None, "auto", 1, shs, sms, False, True, kc6b) == 5
    assert bench.launches_of_group(None, "auto", 3, shs, sms, False, True, kc6b) == 2 + 6 + 3
    assert bench.launches_of_group(None, "auto", 2, shs, sms, False, False, kc6) == 8
    assert bench.launches_of_group(None, "shuffle", 3, shs, sms, False, False, kc6) == 8 + 5
    assert bench.launches_of_group(None, "auto", 3, shs, sms, False, False, kc6) == 12  # decode-MMA: 2 per class


def test_decoder_groups_whole_vector_stack():
    """The whole-vector workload groups q, k and v of each layer (one
    exl3_gemm_whole_grouped call) and runs o alone."""
    gemvs = synth.whole_attention_stack()
    g = bench.decoder_groups(gemvs)
    assert len(g) == 16
    for x in g:
        names = [gemvs[i][0].split(".")[1] for i in x]
        assert names in (["q", "k", "v"], ["o"])


def test_reference_config_matches_the_gpu_line():
    """The reference arm's `config` is the GPU arm's (same workload, shapes,
    grouping and call count), built from host information only."""
    from trellis_decode_gemv_gb300 import binding as B
    assert bench.MAX_GROUP == B.MAX_GROUP
    args = bench.argparse.Namespace(prefill="auto", grouping="step", path="auto")
    desc, cfg, gemvs, M = bench.workload("llama8b", 1)
    grouping = bench.resolve_grouping("step", M, False)
    groups = bench.groups_of([tuple(g) for g in gemvs], grouping, bench.MAX_GROUP)
    c = bench.step_config(args, desc, gemvs, M, grouping, groups, "auto")
    assert c["gemvs_per_step"] == 42 and c["packed_bytes_per_step"] == 490733568
    assert c["grouping"] == "step" and c["calls"].endswith("; 1 calls per step")
    assert bench.resolve_grouping("step", 512, False) == "none"
    assert bench.resolve_grouping("step", 1, True) == "class"
