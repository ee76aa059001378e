"""GPU parity of the FP8 (e4m3) Q K^T path against the oracle, through the C ABI.

The quantiser is byte work: its codes and scale must equal the oracle's bit
for bit. The forward with e4m3 Q K^T computes the attention of the
dequantised Q and K (exact: the scales are powers of two) with V, so it is
compared with the oracle run on those dequantised inputs, at the tolerances of
test_gpu_attention.py.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as A
from oracle import fp8 as F

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 1e-2, 1e-3


def _quant_gpu(x):
    from context_document_masked_gb300 import fcp
    out = torch.empty(x.numel(), dtype=torch.uint8, device="cuda")
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    scratch = torch.empty(1, dtype=torch.int32, device="cuda")
    fcp.quant_e4m3(x, out, scale, scratch)
    torch.cuda.synchronize()
    return out.cpu().numpy(), float(scale.item())


@pytest.mark.parametrize("seed,mag", [(0, 1.0), (1, 300.0), (2, 1e-3), (3, 7.0)])
def test_quant_e4m3_bit_exact(cuda, seed, mag):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(4096 * 8, generator=g) * mag)
    x[:64] = x[:64] * 1e-4          # values that become e4m3 subnormals (or zero) after scaling
    x[64] = 0.0
    x[65] = -0.0
    x = x.to(torch.bfloat16)
    codes, scale = _quant_gpu(x.cuda())
    ref_codes, k = F.quantize_tensor(x.to(torch.float64).numpy())
    assert scale == 2.0 ** k
    assert np.array_equal(codes, ref_codes)


@pytest.mark.parametrize("amax_exp", [-119, -120, -126, -130])
def test_quant_e4m3_tiny_amax_keeps_scale_finite(cuda, amax_exp):
    """amax at or below 2^-119: the scale stops at 2^127 on both sides."""
    g = torch.Generator().manual_seed(-amax_exp)
    x = (torch.rand(4096, generator=g) * 2 - 1) * 2.0 ** amax_exp
    x[7] = 2.0 ** amax_exp
    x = x.to(torch.bfloat16)
    codes, scale = _quant_gpu(x.cuda())
    ref_codes, k = F.quantize_tensor(x.to(torch.float64).numpy())
    assert scale == 2.0 ** k and k == 127
    assert np.array_equal(codes, ref_codes)


def _case(D, hq, hkv, d, cp, pol, seed=0):
    from context_document_masked_gb300.session import CPAttention
    T = sum(D)
    q, k, v = synth.make_qkv(T, hq, hkv, d, seed=seed)
    return CPAttention(D, cp, pol, hq, hkv, d), synth.cu_from_lengths(D), q, k, v


CASES = [
    ("ragged_d128_perdoc", synth.random_doc_lengths(1024, seed=7), 4, 2, 128, 4, "perdoc"),
    ("ragged_d128_hybrid", synth.random_doc_lengths(2048, seed=9), 8, 2, 128, 4, "hybrid"),
    ("tiles_edges", [1, 127, 128, 129, 255, 256, 1, 1, 600, 2], 4, 2, 128, 3, "perdoc"),
    ("long_doc_gqa4", [3000, 40, 1, 55], 8, 2, 128, 2, "perdoc"),
    ("mha_d128", synth.random_doc_lengths(1024, seed=14), 4, 4, 128, 2, "perdoc"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_forward_qk8_matches_oracle_on_dequantised_inputs(cuda, case):
    name, D, hq, hkv, d, cp, pol = case
    s, cu, q, k, v = _case(D, hq, hkv, d, cp, pol)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    s.gather(kd, vd)
    out, lse = s.forward_qk8(qd, kd, vd, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    qq = F.dequantized_tensor(q.to(torch.float64).numpy())
    kq = F.dequantized_tensor(k.to(torch.float64).numpy())
    o_ref, lse_ref = A.attention_per_doc(qq, kq, v, cu)
    e_o = float(np.abs(out.cpu().double().numpy() - o_ref).max())
    e_l = float(np.abs(lse.cpu().double().numpy() - lse_ref).max())
    print(f"[err] qk8 O {e_o:.3e} LSE {e_l:.3e}")
    assert e_o <= TOL_O and e_l <= TOL_LSE


def test_forward_qk8_key_blocks_and_one_shard(cuda):
    """The e4m3 path through the key-block and one-shard forms as well."""
    name, D, hq, hkv, d, cp, pol = CASES[1]
    s, cu, q, k, v = _case(D, hq, hkv, d, cp, pol)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    qq = F.dequantized_tensor(q.to(torch.float64).numpy())
    kq = F.dequantized_tensor(k.to(torch.float64).numpy())
    s.gather(kd, vd)
    lo, hi = 300, 1500
    out, lse = s.forward_qk8(qd, kd, vd, kv_block=(lo, hi), out_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, l_ref = A.attention_per_doc(qq, kq, v, cu, key_range=(lo, hi))
    lg = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    assert np.abs(lg[fin] - l_ref[fin]).max() <= TOL_LSE
    assert np.abs(out.cpu().double().numpy() - o_ref).max() <= TOL_O
    o_full, l_full = A.attention_per_doc(qq, kq, v, cu)
    out1 = torch.full((s.T, hq, d), float("nan"), device="cuda")
    lse1 = torch.full((hq, s.T), float("nan"), device="cuda")
    for j in range(cp):
        s.gather(kd, vd, shard=j)
        s.forward_qk8(qd, kd, vd, shard=j, out=out1, lse=lse1, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert s.device_status() == 0
    assert np.abs(out1.cpu().double().numpy() - o_full).max() <= TOL_O
    assert np.abs(lse1.cpu().double().numpy() - l_full).max() <= TOL_LSE


def test_forward_qk8_rejects_d64(cuda):
    from context_document_masked_gb300 import fcp
    s, cu, q, k, v = _case([64, 64], 4, 2, 64, 2, "perdoc")
    with pytest.raises(fcp.FcpError):
        s.forward_qk8(q.cuda(), k.cuda(), v.cuda())
