"""mha_layer_fwd_host: the self-attention sublayer on pinned host x and y, the batch cut into
slices whose copies overlap the computation.  Each result must equal mha_layer_fwd run on the
same slices on the device bit for bit, and meet the oracle's bound."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity_util import assert_bf16_close, assert_f32_close

import transformer_head_scaled_04_gb300 as mha

pytestmark = pytest.mark.gpu


def _per_slice_on_device(t, w, key_len, chunks):
    """mha_layer_fwd on each slice of the batch, on device tensors."""
    Bc = -(-w.B // min(chunks, w.B))
    ys = []
    for b0 in range(0, w.B, Bc):
        kl = None if key_len is None else key_len[b0:b0 + Bc]
        ys.append(mha.mha_layer(t["x_q"][b0:b0 + Bc], None, t["W_qkv"], t["b_qkv"], t["W_o"],
                                t["b_o"], t["gamma"], t["beta"], w.H, w.mask, kl))
    return torch.cat(ys).cpu()


@pytest.mark.parametrize("name,B,chunks", [
    ("enc_self_base_b32_n128", 32, 4),
    ("enc_self_base_b32_n128", 7, 3),      # a last slice of one sequence
    ("dec_causal_base_b32_n256", 6, 1),
    ("dec_causal_base_b32_n256", 5, 8),    # more slices asked for than sequences
])
def test_layer_host_matches_device_slices(name, B, chunks):
    w = dataclasses.replace(si.WORKLOADS[name], B=B)
    inp = si.draw_layer(w, affine=True)
    dev = torch.device("cuda", 0)
    t = {k: (None if v is None else torch.from_numpy(v).to(dev, torch.bfloat16))
         for k, v in inp.items() if k != "key_len"}
    x_host = t["x_q"].cpu().pin_memory()
    y = mha.mha_layer_host(x_host, t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"], t["gamma"],
                           t["beta"], w.H, w.mask, chunks=chunks)
    ref_dev = _per_slice_on_device(t, w, None, chunks)
    assert torch.equal(y, ref_dev)
    ref = oracle.mha_layer_ref(inp["x_q"], None, inp["W_qkv"], inp["b_qkv"], inp["W_o"],
                               inp["b_o"], inp["gamma"], inp["beta"], w.H, w.mask)
    assert_bf16_close(y.float().numpy(), ref, f"host-buffer sublayer {name} B={B} chunks={chunks}")
    assert mha.device_status() == 0


def test_layer_host_key_padding_and_f32():
    w = si.Workload("t", "layer", "bf16", B=5, H=4, Nq=200, Nk=200, mask="key_padding", seed=61)
    inp = si.draw_layer(w, affine=True)
    inp["key_len"] = np.array([200, 0, 1, 129, 64], np.int32)
    dev = torch.device("cuda", 0)
    t = {k: (None if v is None else torch.from_numpy(v).to(dev, torch.bfloat16))
         for k, v in inp.items() if k != "key_len"}
    kl = torch.from_numpy(inp["key_len"]).to(dev)
    y = mha.mha_layer_host(t["x_q"].cpu().pin_memory(), t["W_qkv"], t["b_qkv"], t["W_o"],
                           t["b_o"], t["gamma"], t["beta"], w.H, "key_padding", kl, chunks=2)
    assert torch.equal(y, _per_slice_on_device(t, w, kl, 2))
    ref = oracle.mha_layer_ref(inp["x_q"], None, inp["W_qkv"], inp["b_qkv"], inp["W_o"],
                               inp["b_o"], inp["gamma"], inp["beta"], w.H, "key_padding",
                               inp["key_len"])
    assert_bf16_close(y.float().numpy(), ref, "host-buffer sublayer key padding")
    wf = si.Workload("t", "layer", "f32", B=3, H=2, Nq=40, Nk=40, seed=62)
    inp = si.draw_layer(wf, affine=True)
    tf = {k: (None if v is None else torch.from_numpy(v).to(dev, torch.float32))
          for k, v in inp.items() if k != "key_len"}
    y = mha.mha_layer_host(tf["x_q"].cpu().pin_memory(), tf["W_qkv"], tf["b_qkv"], tf["W_o"],
                           tf["b_o"], tf["gamma"], tf["beta"], wf.H, "none", chunks=2)
    ref = oracle.mha_layer_ref(inp["x_q"], None, inp["W_qkv"], inp["b_qkv"], inp["W_o"],
                               inp["b_o"], inp["gamma"], inp["beta"], wf.H, "none")
    assert_f32_close(y.numpy(), ref, "host-buffer sublayer f32")
    assert mha.device_status() == 0
