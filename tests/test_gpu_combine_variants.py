"""GPU parity of the combine variants against the oracle, bit for bit: the combine of FP8
rows (the FP8 dispatch's own output, and random codes and scales) and the combined top-k
weights. Outputs sit between guard regions."""
import numpy as np
import pytest
import torch

import combine_ep_get_05_gb300 as ep
import oracle
import workloads
from gpu_helpers import SENT_BF16, SENT_F32, check_guards, dev_bf16, gpu_layout, guarded, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ep.build_library()
    ep.lib()


def _gpu_combine_fp8(codes, scales, slot, M, T, H):
    out, bout = guarded((T, H), torch.bfloat16, SENT_BF16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_combine_fp8(codes, scales, slot, M, out, st)
    torch.cuda.synchronize()
    check_guards(bout, out.numel(), SENT_BF16)
    return host_bits(out), int(st.item())


def _gpu_combine_weights(w, slot, M, T, k):
    out, bout = guarded((T, k), torch.float32, SENT_F32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_combine_weights(w, slot, M, out, st)
    torch.cuda.synchronize()
    check_guards(bout, out.numel(), SENT_F32)
    return host_bits(out), int(st.item())


def _fp8_dispatch(w, M):
    topk, lay = gpu_layout(w)
    d = ep.alloc_dispatch(w.R, M, w.H, w.k, fp8=True)
    d.recv_x.fill_(0)
    d.recv_scales.fill_(0)
    ep.dispatch(dev_bf16(w.x), topk, torch.from_numpy(w.topk_w).cuda(), lay, M, fp8=True, out=d)
    return lay, d


@pytest.mark.parametrize("name,over", [
    ("dsv3_fp8", {"T": 1000, "H": 1024}),
    ("dsv3_fp8", {"T": 333, "H": 384}),
    ("dsv3_fp8", {"T": 1, "H": 128}),
    ("dsv3_fp8", {}),  # the full 4096 x 7168 batch
])
def test_combine_fp8_of_the_fp8_dispatch_matches_oracle(name, over):
    w = workloads.make(name, **over)
    M = w.max_tokens
    lay, d = _fp8_dispatch(w, M)
    got, flags = _gpu_combine_fp8(d.recv_x, d.recv_scales, lay.slot, M, w.T, w.H)
    ref, rflags = oracle.combine_fp8(host_bits(d.recv_x), host_bits(d.recv_scales), host_bits(lay.slot), M)
    assert flags == rflags == 0
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("T,H,R,M,cap", [(700, 512, 8, 700, None), (64, 2048, 33, 64, None), (500, 256, 16, 500, 20)])
def test_combine_fp8_random_rows_match_oracle(T, H, R, M, cap):
    rng = np.random.Generator(np.random.PCG64(77 + T))
    slot = np.full((T, R), -1, np.int32)
    cnt = [0] * R
    for t in range(T):
        for r in range(R):
            if rng.random() < 0.4:
                slot[t, r] = cnt[r]
                cnt[r] += 1
    slot[0, :] = -1
    Mx = max(cnt) if cap is None else cap
    codes = rng.integers(0, 256, (R, Mx, H)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3F  # no NaN codes
    scales = np.exp(rng.uniform(-20, 8, (R, Mx, H // 128))).astype(np.float32)
    got, flags = _gpu_combine_fp8(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(),
                                  torch.from_numpy(slot).cuda(), Mx, T, H)
    ref, rflags = oracle.combine_fp8(codes, scales, slot, Mx)
    assert flags == rflags
    assert np.array_equal(got, ref)


def test_combine_fp8_tiny_scales_and_many_ranks_match_oracle():
    """Scales from 2^-150 to 2^-130 (the first term takes its two-instruction form below
    2^-140), zero scales, products that round to +-0 or to subnormals, and R = 100 ranks
    (slot entries past the first 64 are read as the list is built)."""
    T, H, R = 300, 256, 100
    rng = np.random.Generator(np.random.PCG64(4242))
    slot = np.full((T, R), -1, np.int32)
    cnt = [0] * R
    for t in range(T):
        for r in range(R):
            if rng.random() < 0.12:
                slot[t, r] = cnt[r]
                cnt[r] += 1
    M = max(cnt)
    codes = rng.integers(0, 256, (R, M, H)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3F  # no NaN codes
    codes[:, :, ::7] = 0x80  # -0 codes
    scales = np.ldexp(1.0, rng.integers(-150, -129, (R, M, H // 128))).astype(np.float32)
    scales *= rng.uniform(1.0, 2.0, scales.shape).astype(np.float32)
    scales[rng.random(scales.shape) < 0.1] = 0.0
    assert (scales[scales > 0] < 2.0 ** -140).any() and (scales >= 2.0 ** -140).any()
    got, flags = _gpu_combine_fp8(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(),
                                  torch.from_numpy(slot).cuda(), M, T, H)
    ref, rflags = oracle.combine_fp8(codes, scales, slot, M)
    assert flags == rflags == 0
    assert np.array_equal(got, ref)
    # the data reaches both signed zeros (a negative fp32 sum below bf16's smallest
    # subnormal rounds to -0) and bf16 subnormals
    assert (ref == 0x0000).any() and (ref == 0x8000).any() and (((ref & 0x7F80) == 0) & ((ref & 0x7F) != 0)).any()


@pytest.mark.parametrize("name,over", [
    ("dsv3", {"T": 1000, "H": 8}),
    ("restripe", {"T": 700, "H": 8}),  # empty (-1) slots
    ("skewed", {"T": 3000, "H": 8}),
    ("dsv3", {"T": 1, "H": 8}),
])
def test_combined_weights_match_oracle_and_router_weights(name, over):
    w = workloads.make(name, **over)
    L = oracle.layout(w.topk_idx, w.E, w.R)
    M = int(L["tokens_per_rank"].max()) or 1
    topk, lay = gpu_layout(w)
    d = ep.alloc_dispatch(w.R, M, w.H, w.k)
    ep.dispatch(dev_bf16(w.x), topk, torch.from_numpy(w.topk_w).cuda(), lay, M, out=d)
    got, flags = _gpu_combine_weights(d.recv_topk_w, lay.slot, M, w.T, w.k)
    ref, rflags = oracle.combine_weights(host_bits(d.recv_topk_w), host_bits(lay.slot), M)
    assert flags == rflags == 0
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    exp = np.where((w.topk_idx >= 0) & (w.topk_idx < w.E), w.topk_w, np.float32(0)).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), exp.view(np.uint32))


def test_combined_weights_random_rows_and_capacity():
    rng = np.random.Generator(np.random.PCG64(78))
    T, R, k, M = 900, 64, 8, 40
    slot = np.full((T, R), -1, np.int32)
    cnt = [0] * R
    for t in range(T):
        for r in rng.choice(R, size=rng.integers(0, 9), replace=False):
            slot[t, r] = cnt[r]
            cnt[r] += 1
    w = (rng.standard_normal((R, M, k)) * 10.0 ** rng.integers(-4, 5, (R, M, k))).astype(np.float32)
    got, flags = _gpu_combine_weights(torch.from_numpy(w).cuda(), torch.from_numpy(slot).cuda(), M, T, k)
    ref, rflags = oracle.combine_weights(w, slot, M)
    assert rflags == oracle.FLAG_CAPACITY and flags == rflags
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_combine_variants_reject_bad_arguments():
    t = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = ep.lib()
    assert lib.ep_combine_fp8(None, None, None, 4, 100, 2, 4, None, None, None) == ep.EP_ERR_INVALID  # H % 128
    assert lib.ep_combine_weights(None, None, 4, 33, 2, 4, None, None, None) == ep.EP_ERR_INVALID  # k > 32
    assert lib.ep_combine_fp8(None, None, None, 0, 128, 2, 4, None, None, None) == ep.EP_OK  # empty batch
    del t
