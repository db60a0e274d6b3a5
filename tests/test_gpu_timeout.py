"""The grouped GEMM's failure detection, exercised without faulting or hanging anything:
every pipeline wait of the kernels is bounded, and a wait that runs out sets
MOE_DEV_PIPELINE_TIMEOUT in the device status word, makes every role of the CTA (and of
its partner CTA, for the BF16 computation on SM pairs) leave its loop, waits for the copies and MMAs
still in flight, frees the tensor memory and returns.  A test-only export of the library
(absent from the public header) runs one grouped GEMM with a wait limit of a few
nanoseconds, so that the first wait that is not satisfied at once runs out; the call must
return with the status bit set, and the next ordinary call on the same stream must give
the same output, bit for bit, as a fresh run."""
import ctypes

import numpy as np
import pytest
import torch

import combine_moe_route_softmax_gb300 as moe
from gpu_helpers import bits, need_gpu
from oracle import moe_ref as ref
from oracle.formats import bf16_bits_to_f32

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p
I32 = ctypes.c_int


def wait_limit_fn():
    f = moe.lib().moe_testing_grouped_gemm_wait_limit
    f.restype = I32
    f.argtypes = [P, P, P, I32, I32, I32, I32, P, P, I32, P, P, I32, I32, P, P, P, P, ctypes.c_ulonglong, I32, P]
    return f


def ptr(t):
    return None if t is None else t.data_ptr()


def run(f, a, a_s, cu, w, w_s, dtype, epi, out, out_s, st, limit_ns, pairs):
    stream = torch.cuda.current_stream().cuda_stream
    rc = f(ptr(a), ptr(a_s), ptr(cu), cu.numel() - 1, a.shape[0], a.shape[1], w.shape[1], ptr(w), ptr(w_s),
           w.shape[0], None, None, dtype, epi, ptr(out), ptr(out_s), ptr(st), None, limit_ns, int(pairs), stream)
    assert rc == 0, rc


@pytest.mark.parametrize("kind", ["bf16", "bf16-pairs", "e4m3"])
@pytest.mark.parametrize("swiglu", [False, True], ids=["plain", "swiglu"])
def test_wait_that_runs_out_aborts_cleanly(kind, swiglu):
    need_gpu()
    fp8, pairs = kind == "e4m3", kind == "bf16-pairs"
    f = wait_limit_fn()
    g = torch.Generator().manual_seed(5)
    cu = torch.tensor([0, 300, 300, 1000], dtype=torch.int32)
    k, n, E = 1024, 512, 3
    a = torch.randn(1100, k, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, n, k, generator=g) / k ** 0.5).to(torch.bfloat16)
    cols = n // 2 if swiglu else n
    epi = moe.MOE_EPI_SWIGLU if swiglu else moe.MOE_EPI_NONE
    if fp8:
        qa, sa = ref.act_quant_1x128(bf16_bits_to_f32(bits(a)))
        qw, sw = zip(*[ref.weight_quant_128x128(bf16_bits_to_f32(bits(w[i]))) for i in range(E)])
        A, A_s = torch.from_numpy(qa).cuda(), torch.from_numpy(sa).cuda()
        W, W_s = torch.from_numpy(np.stack(qw)).cuda(), torch.from_numpy(np.stack(sw)).cuda()
        dtype = moe.MOE_E4M3
    else:
        A, A_s, W, W_s, dtype = a.cuda(), None, w.cuda(), None, moe.MOE_BF16
    if fp8 and swiglu:
        mk_out = lambda: torch.zeros(1100, cols, dtype=torch.uint8, device="cuda")
        mk_s = lambda: torch.zeros(1100, cols // 128, dtype=torch.float32, device="cuda")
    else:
        mk_out = lambda: torch.zeros(1100, cols, dtype=torch.bfloat16, device="cuda")
        mk_s = lambda: None
    cu_d = cu.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # a fresh run with the built-in limit
    ref_out, ref_s = mk_out(), mk_s()
    run(f, A, A_s, cu_d, W, W_s, dtype, epi, ref_out, ref_s, st, 2_000_000_000, pairs)
    torch.cuda.synchronize()
    assert st.item() == 0
    # a limit of a few nanoseconds: the first wait that is not satisfied at once runs out
    out, out_s = mk_out(), mk_s()
    run(f, A, A_s, cu_d, W, W_s, dtype, epi, out, out_s, st, 4, pairs)
    torch.cuda.synchronize()       # the call returned: nothing waits forever
    assert st.item() & moe.MOE_DEV_PIPELINE_TIMEOUT
    # the next ordinary call on the same stream is unaffected
    st.zero_()
    out2, out2_s = mk_out(), mk_s()
    run(f, A, A_s, cu_d, W, W_s, dtype, epi, out2, out2_s, st, 2_000_000_000, pairs)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(out2.view(torch.uint8), ref_out.view(torch.uint8))
    if ref_s is not None:
        assert torch.equal(out2_s, ref_s)


@pytest.mark.parametrize("pairs", [False, True], ids=["cta", "pairs"])
@pytest.mark.parametrize("swiglu", [False, True], ids=["plain", "swiglu"])
def test_wait_that_runs_out_aborts_cleanly_with_streaming(swiglu, pairs):
    """The same on a launch large enough to split its CTAs: segments of at most 32 rows on
    the streaming CTAs, whose two pipeline lanes (two TMA threads, two MMA threads) each
    drain their own stages and MMAs on the way out."""
    need_gpu()
    f = wait_limit_fn()
    rng = np.random.default_rng(41 + swiglu + 2 * pairs)
    counts = list(rng.integers(0, 33, 60)) + [3900 + int(rng.integers(0, 100)) for _ in range(10)]
    rng.shuffle(counts)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32)
    k, n, E = 256, 2048, len(counts)
    g = torch.Generator().manual_seed(43)
    a = torch.randn(int(cu[-1]), k, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(E, n, k, generator=g) / k ** 0.5).to(torch.bfloat16).cuda()
    cols = n // 2 if swiglu else n
    epi = moe.MOE_EPI_SWIGLU if swiglu else moe.MOE_EPI_NONE
    mk = lambda: torch.zeros(a.shape[0], cols, dtype=torch.bfloat16, device="cuda")
    cu_d = cu.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_out = mk()
    run(f, a, None, cu_d, w, None, moe.MOE_BF16, epi, ref_out, None, st, 2_000_000_000, pairs)
    torch.cuda.synchronize()
    assert st.item() == 0
    out = mk()
    run(f, a, None, cu_d, w, None, moe.MOE_BF16, epi, out, None, st, 4, pairs)
    torch.cuda.synchronize()       # the call returned: nothing waits forever
    assert st.item() & moe.MOE_DEV_PIPELINE_TIMEOUT
    st.zero_()
    out2 = mk()
    run(f, a, None, cu_d, w, None, moe.MOE_BF16, epi, out2, None, st, 2_000_000_000, pairs)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(out2.view(torch.int16), ref_out.view(torch.int16))
