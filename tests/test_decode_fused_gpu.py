"""GPU parity of the decode whose split partials are merged inside a thread-block
cluster (one launch, no workspace), against the fp64 oracle and the two-kernel
path.  Cache rows past each sequence length hold NaN."""
import math

import numpy as np
import pytest
import torch

import gqa_attention_gb300 as g
from gqa_attention_gb300 import inputs

from parity import assert_parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_attention_gb300 import build

    build.build()
    g.load()
    yield
    assert g.gqa_last_device_error() == g.GQA_OK


def _fused(q, k, v, lens):
    out, lse = g.decode_fused(q.to(DEV), k.to(DEV), v.to(DEV), lens.to(DEV))
    torch.cuda.synchronize()
    return out, lse


def test_cluster_size_on_this_device():
    c = g.gqa_attn_decode_fused_splits(1, 64, 8, 128)
    assert c in (8, 16)
    assert g.gqa_attn_decode_fused_splits(1, 64, 8, 96) == 0  # head dim
    assert g.gqa_attn_decode_fused_splits(1, 34, 2, 128) == 0  # G = 17


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("G", [1, 4, 8, 16])
@pytest.mark.parametrize("ctx", [1, 63, 65, 700, 1025, 5000])
def test_small_shapes(oracle_mod, d, G, ctx):
    # short contexts leave most of the cluster's splits empty
    H_kv = 2
    q, k, v, lens = inputs.decode_inputs(1, G * H_kv, H_kv, d, ctx, seed=ctx + 3 * G + d)
    ref_o, ref_l = oracle_mod.decode(q, k, v, lens, 1 / math.sqrt(d))
    out, lse = _fused(q, k, v, lens)
    assert_parity(out, lse, ref_o, ref_l, f"fused d={d} G={G} ctx={ctx}")


@pytest.mark.parametrize("B,S_max,lens", [(3, 300, [1, 299, 300]), (4, 1000, [64, 65, 999, 128]),
                                          (2, 5000, [4097, 17])])
def test_ragged_batches_match_oracle_and_two_kernel_path(oracle_mod, B, S_max, lens):
    q, k, v, sl = inputs.decode_inputs(B, 32, 4, 128, S_max, seed=B + 40, seq_lens=lens)
    ref_o, ref_l = oracle_mod.decode(q, k, v, sl, 1 / math.sqrt(128))
    out, lse = _fused(q, k, v, sl)
    assert_parity(out, lse, ref_o, ref_l, f"fused B={B} lens={lens}")
    # the same merge with the cluster's split count through the two kernels
    c = g.gqa_attn_decode_fused_splits(B, 32, 4, 128)
    out2, lse2 = g.decode(q.to(DEV), k.to(DEV), v.to(DEV), sl.to(DEV), n_split=c)
    torch.cuda.synchronize()
    assert (out.float() - out2.float()).abs().max().item() <= 2 ** -7
    assert (lse - lse2).abs().max().item() <= 1e-5


def test_deterministic_across_runs():
    q, k, v, lens = inputs.decode_inputs(1, 64, 8, 128, 4096, seed=12)
    a = _fused(q, k, v, lens)
    b = _fused(q, k, v, lens)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])


def test_outputs_stay_inside_their_buffers():
    B, H_q, H_kv, d = 2, 16, 2, 128
    q, k, v, lens = inputs.decode_inputs(B, H_q, H_kv, d, 700, seed=6, seq_lens=[700, 3])
    pad = 4096
    out_buf = torch.full((B * H_q * d + 2 * pad,), 7.0, dtype=torch.bfloat16, device=DEV)
    lse_buf = torch.full((B * H_q + 2 * pad,), 7.0, dtype=torch.float32, device=DEV)
    out = out_buf[pad: pad + B * H_q * d].view(B, H_q, d)
    lse = lse_buf[pad: pad + B * H_q].view(B, H_q)
    g.decode_fused(q.to(DEV), k.to(DEV), v.to(DEV), lens.to(DEV), out=out, lse=lse)
    torch.cuda.synchronize()
    for buf, n in ((out_buf, B * H_q * d), (lse_buf, B * H_q)):
        assert (buf[:pad].float() == 7.0).all() and (buf[pad + n:].float() == 7.0).all()


def test_bad_seq_len_gives_nan_and_error_word():
    q, k, v, lens = inputs.decode_inputs(2, 8, 2, 64, 128, seed=2)
    lens[1] = 129  # past S_max: caught on the device
    out, lse = _fused(q, k, v, lens)
    assert g.gqa_last_device_error() == g.GQA_ERR_INVALID_ARG
    assert torch.isnan(out[1].float()).all() and torch.isnan(lse[1]).all()
    assert torch.isfinite(out[0].float()).all() and torch.isfinite(lse[0]).all()
    assert g.gqa_last_device_error() == g.GQA_OK


def test_rejects_bad_host_arguments():
    x = torch.empty(64, dtype=torch.bfloat16, device=DEV)
    t = torch.ones(1, dtype=torch.int32, device=DEV)
    f = torch.empty(8, dtype=torch.float32, device=DEV)
    assert g.gqa_attn_decode_fused(x, x, x, t, 1, 4, 8, 2, 96, 0.1, x, f) == g.GQA_ERR_UNSUPPORTED
    assert g.gqa_attn_decode_fused(x, x, x, None, 1, 4, 8, 2, 64, 0.1, x, f) == g.GQA_ERR_INVALID_ARG
    assert g.gqa_attn_decode_fused(x, x, x, t, 1, 4, 8, 3, 64, 0.1, x, f) == g.GQA_ERR_INVALID_ARG


@pytest.mark.parametrize("cfg", inputs.DECODE_CONFIGS, ids=lambda c: c.name)
def test_full_size_workloads(oracle_mod, cfg):
    """The three decode workloads at full size."""
    q, k, v, lens = inputs.decode_inputs_for(cfg, seed=0)
    ref_o, ref_l = oracle_mod.decode(q, k, v, lens, cfg.scale)
    out, lse = _fused(q, k, v, lens)
    assert_parity(out, lse, ref_o, ref_l, "fused " + cfg.name)
    assert np.isfinite(lse.cpu().numpy()).all()
