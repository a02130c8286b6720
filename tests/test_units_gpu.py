"""PTX building blocks of the bf16 kernel, one at a time, on the GPU.

Each check uses the same tile geometry, descriptors and encodings as the
attention kernel: a wrong swizzle, descriptor bit field or instruction
encoding shows up here as a wrong number."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DS = [16, 32, 64, 128]


def _bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def expected_swizzled_image(x: np.ndarray, d: int) -> np.ndarray:
    """Shared-memory image of a [128][d] bf16 tile loaded as boxes of
    min(d, 64) columns with the swizzle of the box-row width: 16-byte chunk
    bits [4, 4+B) of every byte offset are XORed with bits [7, 7+B), B = 1, 2, 3
    for 32-, 64-, 128-byte rows."""
    box_x = min(d, 64)
    row_bytes = box_x * 2
    nbox = d // box_x
    B = {32: 1, 64: 2, 128: 3}[row_bytes]
    mask = ((1 << B) - 1) << 4
    img = np.zeros(128 * d, dtype=np.uint16)
    r = np.arange(128)[:, None]
    c = np.arange(box_x)[None, :]
    for bx in range(nbox):
        lin = bx * 128 * row_bytes + r * row_bytes + c * 2
        phys = lin ^ ((lin >> 3) & mask)
        img[(phys // 2).ravel()] = x[:, bx * box_x:(bx + 1) * box_x].ravel()
    return img


@pytest.mark.parametrize("d", DS)
def test_tma_swizzled_tile(cuda_lib, d):
    fa = cuda_lib
    x = _bf16((1, 1, 128, d), seed=d).cuda()
    out = torch.zeros(128 * d, dtype=torch.int16, device="cuda")
    assert fa.fa_unit_tma(x, out, d) == 0
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    want = expected_swizzled_image(x.cpu().view(torch.int16).numpy().view(np.uint16)[0, 0], d)
    assert np.array_equal(got, want)
    assert fa.fa_debug_sync_check() == 0


@pytest.mark.parametrize("d", DS)
def test_mma_qk_kmajor(cuda_lib, d):
    fa = cuda_lib
    q = _bf16((1, 1, 128, d), seed=10 + d).cuda()
    k = _bf16((1, 1, 128, d), seed=20 + d).cuda()
    s = torch.zeros(128, 128, dtype=torch.float32, device="cuda")
    assert fa.fa_unit_qk(q, k, s, d) == 0
    torch.cuda.synchronize()
    qd, kd = q[0, 0].double().cpu(), k[0, 0].double().cpu()
    ref = qd @ kd.T
    bound = 1e-5 * (qd.abs() @ kd.abs().T) + 1e-6
    err = (s.double().cpu() - ref).abs()
    assert torch.all(err <= bound), f"max err {err.max().item():.3g}"
    assert fa.fa_debug_sync_check() == 0


def test_tmem_store_load_round_trip(cuda_lib):
    """P rounded to bf16, two per 32-bit column (even key in the low half),
    written with tcgen05.st and read back with tcgen05.ld."""
    fa = cuda_lib
    g = torch.Generator().manual_seed(3)
    p = torch.rand((128, 128), generator=g).cuda()
    v = _bf16((1, 1, 128, 128), seed=4).cuda()
    o = torch.zeros((128, 64), dtype=torch.float32, device="cuda")
    assert fa.fa_unit_pv(p, None, v, o, 128, mode=3) == 0
    torch.cuda.synchronize()
    words = o.cpu().view(torch.int32).numpy().view(np.uint32)
    pb = p.cpu().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).astype(np.uint32)
    want = pb[:, 0::2] | (pb[:, 1::2] << 16)
    assert np.array_equal(words, want)


@pytest.mark.parametrize("d", DS)
def test_mma_pv_smem_a_mnmajor_b(cuda_lib, d):
    """P from shared memory (K-major, as Q): checks the MN-major V descriptor."""
    fa = cuda_lib
    g = torch.Generator().manual_seed(50 + d)
    pb = torch.rand((128, 128), generator=g).to(torch.bfloat16).cuda()
    v = _bf16((1, 1, 128, d), seed=60 + d).cuda()
    o = torch.full((128, d), float("nan"), dtype=torch.float32, device="cuda")
    assert fa.fa_unit_pv(None, pb, v, o, d, mode=2) == 0
    torch.cuda.synchronize()
    ref = pb.double().cpu() @ v[0, 0].double().cpu()
    bound = 1e-5 * (pb.double().cpu().abs() @ v[0, 0].double().cpu().abs()) + 1e-6
    err = (o.double().cpu() - ref).abs()
    assert torch.all(err <= bound), f"max err {err.max().item():.3g}"
    assert fa.fa_debug_sync_check() == 0


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("d", DS)
def test_mma_pv_tmem_a_mnmajor_b(cuda_lib, d, mode):
    fa = cuda_lib
    g = torch.Generator().manual_seed(30 + d)
    p = torch.rand((128, 128), generator=g).cuda()
    v = _bf16((1, 1, 128, d), seed=40 + d).cuda()
    pb = p.to(torch.bfloat16).double().cpu()
    vd = v[0, 0].double().cpu()
    ref = pb @ vd
    bound = 1e-5 * (pb.abs() @ vd.abs()) + 1e-6
    for _ in range(3 if mode else 1):
        o = torch.full((128, d), float("nan"), dtype=torch.float32, device="cuda")
        assert fa.fa_unit_pv(p, None, v, o, d, mode=mode) == 0
        torch.cuda.synchronize()
        err = (o.double().cpu() - ref).abs()
        assert torch.all(err <= bound), f"max err {err.max().item():.3g}"
    assert fa.fa_debug_sync_check() == 0


def test_bounded_wait_gives_up_and_reports(cuda_lib):
    """A wait on a barrier that nothing arrives on ends after its budget (about
    2 ms here), the timeout is reported once through fa_debug_sync_check, and
    the context stays usable afterwards."""
    fa = cuda_lib
    assert fa.fa_debug_sync_check() == 0
    gave_up = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert fa.fa_unit_timeout(1 << 22, gave_up) == 0
    torch.cuda.synchronize()
    assert gave_up.item() == 128
    assert fa.fa_debug_sync_check() == fa.FA_ERR_TIMEOUT
    assert fa.fa_debug_sync_check() == 0  # read-and-clear
    q = _bf16((1, 2, 256, 64), seed=5).cuda()
    o, lse = fa.fwd(q, q, q, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_debug_sync_check() == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_pipe_rate_probe_measures_plausible_rates(cuda_lib):
    """The probe behind the exp and fp32 rooflines: one CTA per SM, every CTA
    reports a clock span, and the rates per clock per SM lie inside what the
    units can deliver (at most 32 lanes x 4 SMSPs per clock; ex2 on the
    special-function unit well below the FMA rate)."""
    fa = cuda_lib
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sink = torch.zeros(512, dtype=torch.float32, device="cuda")
    cycles = torch.zeros(sms, dtype=torch.int64, device="cuda")
    iters = 1 << 10
    rates = {}
    for kind, per_thread in ((0, 8), (1, 8), (2, 4)):
        for _ in range(2):
            assert fa.fa_unit_pipe_rate(kind, iters, sms, sink, cycles) == 0
        torch.cuda.synchronize()
        c = cycles.cpu()
        assert bool((c > 0).all())
        rates[kind] = float((512 * per_thread * iters / c.double()).median())
    assert fa.fa_debug_sync_check() == 0
    assert 4.0 <= rates[0] <= 64.0            # ex2 instructions per clock per SM
    assert 32.0 <= rates[1] <= 128.0          # scalar FMA instructions
    assert 16.0 <= rates[2] <= 64.0           # paired FMA instructions (two FMAs each)
    assert rates[0] < rates[1]
