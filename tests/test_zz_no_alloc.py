"""aqfq_scale_grad_noalloc: the scale gradient for callers that cannot
allocate device memory (for example a plugin whose host framework owns every
byte of device memory, or a path where a synchronising cudaMalloc is not
allowed).  Through the C ABI, its output must match aqfq_scale_grad with a
caller-provided workspace, on two calls in a row (the built-in scratch is
shared and reused), and sizes beyond its 128 KiB scratch are rejected.  The
cases cover every reduction that takes its scratch from the built-in array:
per-tensor, NVFP4 tensor scale and per-head."""
import ctypes

import numpy as np
import pytest
import torch

from learnable_scale_fake_gb300 import aqfq, synth
from paritylib import assert_grad_close, dev, oracle_grad

pytestmark = pytest.mark.gpu

Q = aqfq.qspec
CASES = [
    ("nvfp4_dynamic", Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16, mode=aqfq.SCALE_DYNAMIC_BLOCK),
     (2, 96, 1024)),
    ("fp8_per_tensor", Q(aqfq.FP8_E4M3, aqfq.PER_TENSOR), (3, 80, 512)),
    ("nvfp4_learned", Q(aqfq.NVFP4, aqfq.PER_GROUP, group=16), (2, 33, 208)),
    # per-head partial sums: 64 * 4 * 128 / 16 = 2048 threads' doubles in the scratch
    ("fp8_per_head", Q(aqfq.FP8_E4M3, aqfq.PER_HEAD), (64, 4, 128)),
]


@pytest.mark.parametrize("name,sp,shape", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_entry(name, sp, shape):
    d = dev()
    B, R, K = shape
    x = synth.normal_outliers_bf16(shape, 0.02, 1e-2, 30.0, seed=91)
    dy = synth.normal_bf16(shape, 1.0, seed=92)
    dyn = sp.fmt == aqfq.NVFP4 and sp.mode == aqfq.SCALE_DYNAMIC_BLOCK
    n = aqfq.scale_numel(sp, B, R, K)
    s = synth.loguniform_f32((n,), 2e-5, 2e-4, seed=93) if n else None
    if sp.fmt == aqfq.NVFP4 and not dyn:
        s = synth.loguniform_f32((n,), 2e-3, 2e-2, seed=93)
    ts = synth.loguniform_f32((B,), 2e-6, 1e-5, seed=94) if sp.fmt == aqfq.NVFP4 else None
    xd, dyd = x.to(d), dy.to(d)
    sd = None if s is None else s.to(d)
    tsd = None if ts is None else ts.to(d)

    def out():
        return torch.zeros(B if dyn else n, device=d)

    # the existing entry point with a caller-provided workspace
    ref = out()
    wsb = aqfq.aqfq_scale_grad_workspace_bytes(sp, B, R, K)
    ws = torch.empty(max(1, wsb // 8), dtype=torch.float64, device=d) if wsb else None
    kw = {"dtensor_scale": ref} if dyn else {"dscale": ref}
    aqfq.aqfq_scale_grad(sp, xd, dyd, sd, tsd, workspace=ws, **kw)
    torch.cuda.synchronize()
    orc = oracle_grad(sp, x, dy, s, ts)
    r_abs = orc["dtensor_scale_abs"] if dyn else orc["dscale_abs"]
    r_val = orc["dtensor_scale"] if dyn else orc["dscale"]
    assert_grad_close(ref.cpu().numpy(), r_val, r_abs)
    # the allocation-free entry, twice in a row through the C ABI
    L = aqfq.lib()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        got = out()
        p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
        rc = L.aqfq_scale_grad_noalloc(ctypes.byref(sp), p(xd), p(dyd), B, R, K, p(sd), p(tsd),
                                       None if dyn else p(got), p(got) if dyn else None, None, 0, st)
        torch.cuda.synchronize()
        assert rc == 0, aqfq.STATUS.get(rc, rc)
        assert_grad_close(got.cpu().numpy(), ref.cpu().numpy().astype(np.float64), r_abs)
        assert_grad_close(got.cpu().numpy(), r_val, r_abs)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    dev()
    sp = Q(aqfq.FP8_E4M3, aqfq.PER_HEAD)
    # per-head partial sums of [65536 tokens, 32 heads, 128] exceed 128 KiB
    assert aqfq.aqfq_scale_grad_workspace_bytes(sp, 65536, 32, 128) > (128 << 10)
    L = aqfq.lib()
    A = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    rc = L.aqfq_scale_grad_noalloc(ctypes.byref(sp), A, A, 65536, 32, 128, A, None, A, None, None,
                                   0, None)
    assert rc == 5  # AQFQ_ERR_WORKSPACE
