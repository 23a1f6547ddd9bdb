"""GPU parity at the full sizes of the measured workloads, in the launch
configuration the benchmark times (splits sized to one wave, fused split-K
merge, CUDA-graph replay of each decode step). The oracle recomputes sampled
(layer, sequence) outputs from its own contiguous histories; INT8 pools are
compared with the oracle's codes and scales byte for byte."""

import gc

import numpy as np
import pytest
import torch

from harness import Workload, assert_close
from libpkv import ensure_built

pytestmark = pytest.mark.gpu
STEPS = 3


@pytest.fixture(autouse=True)
def _lib_and_cleanup():
    ensure_built()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _check(w: Workload, layers, seqs, reps=(0,)):
    outs = [w.step().float().cpu().numpy() for _ in range(STEPS)]
    assert w.error_bits() == 0
    for li in layers:
        for i in seqs:
            for rep in reps:
                ref = w.oracle_steps(li, i, STEPS, rep)
                for t in range(STEPS):
                    assert_close(outs[t][li * w.R + rep, i], ref[t], f"layer {li} seq {i} rep {rep} step {t}")
            w.check_pool_bytes(li, i, w.prior[i] + STEPS)


def test_tts_talker_28_layers_8000_tokens_int8():
    w = Workload(seed=1235, num_layers=28, prior=[8000] * 4, Hq=16, Hkv=8, d=128, bs=16, num_blocks=2048, int8=True,
                 head_scale=True, split_tokens="auto", max_blocks=-(-(8000 + 64) // 16), graph=True)
    assert w.split_tokens > 0
    _check(w, layers=(0, 27), seqs=range(4))


def test_mha7b_32_layers_100x1024_bf16():
    w = Workload(seed=1236, num_layers=32, prior=[1024] * 100, Hq=32, Hkv=32, d=128, bs=16, num_blocks=8192,
                 int8=False, split_tokens="auto", max_blocks=-(-(1024 + 64) // 16), graph=True)
    _check(w, layers=(0, 31), seqs=(0, 41, 99))


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
def test_long_context_8x32768_split_k(int8):
    w = Workload(seed=1237, num_layers=1, prior=[32768] * 8, Hq=32, Hkv=8, d=128, bs=64, num_blocks=4200, int8=int8,
                 outliers=True, split_tokens="auto", max_blocks=-(-(32768 + 64) // 64), graph=True, repeat=32)
    assert w.split_tokens > 0
    _check(w, layers=(0,), seqs=(0, 5), reps=(0, 31))
