"""The step before attention on the GPU (Q/K RMSNorm, partial RoPE, KV write)
against the FP64 oracle.  Elementwise, FP32 with one BF16 rounding: every output
is within one BF16 ulp of the oracle's correctly rounded value and almost all are
identical; copies (gate, V) are exact; pool rows other than the new slots are
untouched.  A prep -> decode test checks the two entry points composed."""
import numpy as np
import pytest
import torch

import oracle
from canary import Guarded, check_all
from gated_gqa_attention_gb300 import workloads

pytestmark = pytest.mark.gpu
D = 256


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def tb(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def ulp_diff(a, b):
    """Distance in BF16 codes (same sign assumed for nonzero pairs)."""
    ia = a.astype(np.int32)
    ib = b.astype(np.int32)
    ia = np.where(ia & 0x8000, 0x8000 - ia, ia)
    ib = np.where(ib & 0x8000, 0x8000 - ib, ib)
    return np.abs(ia - ib)


def make(B, Hq, Hkv, rope_dim, seed, slots_n=300):
    rng = np.random.default_rng(seed)
    f = lambda *s: torch.from_numpy(rng.standard_normal(s).astype(np.float32)).to(torch.bfloat16)
    qgkv = f(B, (2 * Hq + 2 * Hkv) * D) * 2
    wq = torch.from_numpy(rng.uniform(0.5, 1.5, D).astype(np.float32)).to(torch.bfloat16)
    wk = torch.from_numpy(rng.uniform(0.5, 1.5, D).astype(np.float32)).to(torch.bfloat16)
    theta = rng.uniform(0, 6.3, (B, max(rope_dim // 2, 1)))[:, :rope_dim // 2]
    ang = np.concatenate([theta, theta], axis=1)
    cos = torch.from_numpy(np.cos(ang).astype(np.float32)).to(torch.bfloat16)
    sin = torch.from_numpy(np.sin(ang).astype(np.float32)).to(torch.bfloat16)
    slots = torch.from_numpy(rng.permutation(slots_n)[:B].astype(np.int32))
    kp, vp = f(slots_n, Hkv, D), f(slots_n, Hkv, D)
    return qgkv, wq, wk, cos, sin, slots, kp, vp


@pytest.mark.parametrize("B,Hq,Hkv,rope_dim,norm", [
    (1, 16, 2, 64, True), (7, 16, 2, 0, True), (7, 16, 2, 256, False), (224, 16, 2, 64, True),
    (5, 6, 2, 128, True), (3, 32, 4, 16, True)])
def test_prep_matches_oracle(gda, B, Hq, Hkv, rope_dim, norm):
    qgkv, wq, wk, cos, sin, slots, kp, vp = make(B, Hq, Hkv, rope_dim, seed=B + Hq + rope_dim)
    ref_q, ref_g, ref_kp, ref_vp = oracle.qk_norm_rope_kv_write(
        qgkv, wq if norm else None, wk if norm else None, 1e-6, cos, sin, rope_dim, slots, kp, vp, Hq, Hkv, D)
    # every buffer the kernel writes sits inside 0xFF guard bands (canary.Guarded)
    gk, gv = Guarded.copy_of(kp.cuda()), Guarded.copy_of(vp.cuda())
    gq, gg = Guarded((B, Hq, D), torch.bfloat16), Guarded((B, Hq, D), torch.bfloat16)
    dk, dv = gk.t, gv.t
    q_out, g_out = gda.qk_norm_rope_kv_write(
        qgkv.cuda(), slots.cuda(), dk, dv, Hq, w_q_norm=wq.cuda() if norm else None,
        w_k_norm=wk.cuda() if norm else None, eps=1e-6, cos=cos.cuda() if rope_dim else None,
        sin=sin.cuda() if rope_dim else None, rope_dim=rope_dim, q_out=gq.t, gate_out=gg.t)
    check_all(k_pool=gk, v_pool=gv, q_out=gq, gate_out=gg)
    got_q, got_k, got_v = bits(q_out), bits(dk), bits(dv)
    assert np.array_equal(bits(g_out), ref_g)                 # gate copied
    assert np.array_equal(got_v, ref_vp)                       # V written, rest untouched
    dq = ulp_diff(got_q, ref_q)
    dkk = ulp_diff(got_k, ref_kp)
    assert dq.max() <= 1 and dkk.max() <= 1
    assert (dq == 0).mean() > 0.99 and (dkk == 0).mean() > 0.99
    other = np.setdiff1d(np.arange(kp.shape[0]), slots.numpy())
    assert np.array_equal(got_k[other], bits(kp)[other])       # other K rows untouched


def test_prep_then_decode_is_the_layer(gda):
    """prep (norm + rope + KV write) followed by the gated decode equals the oracle of
    the same two steps, the decode reading the rows prep just wrote."""
    B, Hq, Hkv = 6, 16, 2
    lens = [1, 40, 300, 77, 1024, 5]
    inp = workloads.make(lens, seed=55, layout="perm", pool_slots=3000)
    qgkv, wq, wk, cos, sin, _, _, _ = make(B, Hq, Hkv, 64, seed=56)
    # the new token of each sequence sits in its last position's slot
    ip, ix = inp["kv_indptr"].tolist(), inp["kv_indices"]
    slots = torch.tensor([int(ix[ip[b + 1] - 1]) for b in range(B)], dtype=torch.int32)
    ref_q, ref_g, ref_kp, ref_vp = oracle.qk_norm_rope_kv_write(
        qgkv, wq, wk, 1e-6, cos, sin, 64, slots, inp["k_pool"], inp["v_pool"], Hq, Hkv, D)
    ref = oracle.decode(ref_q, ref_g, ref_kp, ref_vp, inp["kv_indptr"], inp["kv_indices"], inp["scale"])
    dk, dv = inp["k_pool"].cuda(), inp["v_pool"].cuda()
    q_out, g_out = gda.qk_norm_rope_kv_write(qgkv.cuda(), slots.cuda(), dk, dv, Hq, w_q_norm=wq.cuda(),
                                             w_k_norm=wk.cuda(), eps=1e-6, cos=cos.cuda(), sin=sin.cuda(),
                                             rope_dim=64)
    out = gda.decode(q_out, g_out, dk, dv, inp["kv_indptr"].cuda(), inp["kv_indices"].cuda(), scale=inp["scale"])
    torch.cuda.synchronize()
    g = oracle.double_from_bf16(bits(out))
    w = oracle.double_from_bf16(ref.out)
    # prep's outputs may differ from the oracle's by one BF16 ulp, which the decode tolerance absorbs
    assert np.all(np.abs(g - w) <= 4e-3 + 1.6e-2 * np.abs(w))


def test_prep_skips_out_of_range_slots(gda):
    qgkv, wq, wk, cos, sin, slots, kp, vp = make(4, 16, 2, 64, seed=9)
    slots[1] = 300            # == num_slots
    slots[2] = -1
    dk, dv = kp.cuda(), vp.cuda()
    gda.qk_norm_rope_kv_write(qgkv.cuda(), slots.cuda(), dk, dv, 16, w_q_norm=wq.cuda(), w_k_norm=wk.cuda(),
                              cos=cos.cuda(), sin=sin.cuda(), rope_dim=64)
    torch.cuda.synchronize()
    keep = np.setdiff1d(np.arange(300), slots.numpy()[[0, 3]])
    assert np.array_equal(bits(dk)[keep], bits(kp)[keep]) and np.array_equal(bits(dv)[keep], bits(vp)[keep])
