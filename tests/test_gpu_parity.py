"""GPU parity: the library (through the C-ABI) against the fp64 oracle.

Sizes the oracle finishes in seconds are compared element by element over
the whole output; the full-size workloads are compared on sampled lines
(rows for the starting node, columns for the ending node), which the oracle
computes one by one, plus properties that hold at any size (padded pairs
exactly zero, chunked equal to unchunked, run-to-run determinism).
"""
import numpy as np
import pytest

from tests.gpu_cases import assert_close, errors, oracle_out, run_library, select

pytestmark = pytest.mark.gpu

NODES = ("start", "end")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_tiny_f32_full():
    res = run_library("tiny_f32")
    for node in NODES:
        assert_close(res[node], oracle_out("tiny_f32", node), "f32", f"tiny_f32 {node}")


@pytest.mark.parametrize("I", [1, 17, 64, 129, 256])
def test_evoformer_shape_full(I):
    """Evoformer-sized channels; I=256 is the workload itself, the rest are ragged tiles."""
    res = run_library("evoformer_256", I=I)
    for node in NODES:
        assert_close(res[node], oracle_out("evoformer_256", node, I=I), "bf16", f"evoformer I={I} {node}")


@pytest.mark.parametrize("I,n_pad", [(200, 77), (130, 3), (96, 95)])
def test_masked_small_full(I, n_pad):
    res = run_library("masked_768", I=I, n_pad=n_pad)
    for node in NODES:
        want = oracle_out("masked_768", node, I=I, n_pad=n_pad)
        assert_close(res[node], want, "bf16", f"masked I={I} pad={n_pad} {node}")
        valid = np.arange(I) < I - n_pad
        pad_pairs = ~(valid[:, None] & valid[None, :])
        assert np.all(res[node][pad_pairs] == 0.0)


def test_all_tokens_masked_gives_zero():
    res = run_library("masked_768", I=40, n_pad=40)
    for node in NODES:
        assert np.all(res[node] == 0.0)


def _sampled(name, lines, nodes=NODES, key_chunks=1, res=None):
    res = res or run_library(name, nodes=nodes, key_chunks=key_chunks)
    from tests.gpu_cases import inputs
    dtype = inputs(name).workload.dtype
    for node in nodes:
        got = select(res[node], node, lines)
        want = oracle_out(name, node, lines=lines, key_chunks=key_chunks)
        assert_close(got, want, dtype, f"{name} {node} lines={lines}")
    return res


def test_masked_768_sampled():
    lines = [0, 345, 690, 691, 767]          # first, middle, last valid, first pad, last pad
    res = _sampled("masked_768", lines)
    for node in NODES:
        out = res[node]
        assert np.all(out[691:] == 0.0) and np.all(out[:, 691:] == 0.0)


@pytest.mark.slow
def test_complex_2048_sampled():
    lines = [0, 255, 256, 1023, 1600, 2047]  # chain boundaries, first and last
    _sampled("complex_2048", lines)


@pytest.mark.slow
def test_single_chain_2752_unchunked_and_chunked():
    lines = [0, 343, 344, 1376, 2751]        # around the 344-token chunk boundaries
    a = _sampled("single_chain_2752", lines, nodes=("start",), key_chunks=1)
    b = _sampled("single_chain_2752", lines, nodes=("start",), key_chunks=8)
    max_abs, _ = errors(b["start"], a["start"])
    assert max_abs <= 2e-2


@pytest.mark.parametrize("chunks", [3, 8])
def test_chunked_small_full(chunks):
    res = run_library("masked_768", I=150, n_pad=20, key_chunks=chunks)
    for node in NODES:
        assert_close(res[node], oracle_out("masked_768", node, I=150, n_pad=20), "bf16", f"chunks={chunks} {node}")


def test_deterministic():
    res = run_library("evoformer_256", repeat=2)
    for node in NODES:
        a, b = res[node]
        assert np.array_equal(a, b)


def test_simt_path_bf16_small():
    res = run_library("evoformer_256", I=80, force_simt=True)
    assert res["path"] == 0
    for node in NODES:
        assert_close(res[node], oracle_out("evoformer_256", node, I=80), "bf16", f"simt bf16 {node}")


@pytest.mark.parametrize("force_simt", [False, True])
def test_affine_params(force_simt):
    """Non-trivial LayerNorm gamma / beta, gate bias and output bias: every term
    they enter (the folded gamma, the beta offset, b_g, b_o) is exercised."""
    res = run_library("evoformer_256", I=129, force_simt=force_simt, affine=True)
    assert res["path"] == (0 if force_simt else 1)
    for node in NODES:
        want = oracle_out("evoformer_256", node, I=129, affine=True)
        assert_close(res[node], want, "bf16", f"affine params {node} simt={force_simt}")
    res_f32 = run_library("tiny_f32", affine=True)
    for node in NODES:
        assert_close(res_f32[node], oracle_out("tiny_f32", node, affine=True), "f32", f"affine f32 {node}")
