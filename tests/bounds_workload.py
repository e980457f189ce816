"""One fixed GPU workload through the library that TTT_LIBRARY selects
(libttt.so, or libttt_debug.so with TTT_LIBRARY=debug), for
test_debug_bounds_gpu.py, which runs it under both and compares.

    python tests/bounds_workload.py OUT.npz     # outputs + range-check record
    python tests/bounds_workload.py --selftest  # one JSON line

The workload covers every kind of range-checked access: the tensor-core
attention forward and backward at head dims 64, 96 (boxes reaching past the
head dim) and 128 (a 128-row chunk, whose tile pair has an empty second
tile, and a 3B chunk deep in the sequence, the ring wrapping), the
one-query attention of a decode step, and a context's prefill and decode at
the 3B widths (bulk pass, chunk loop, decode steps with their ring rows).
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from long_context_lm_ttt_b300 import inputs  # noqa: E402
from long_context_lm_ttt_b300 import ttt as T  # noqa: E402

# n, H, Hkv, hd, W, pos0, R
ATTN = [
    (128, 4, 2, 128, 300, 256, 512),  # a pair's second tile has no rows
    (200, 4, 2, 64, 1000, 0, 1280),
    (256, 6, 2, 96, 300, 1024, 640),
    (1024, 24, 8, 128, 8192, 40960, 9216),
]
DECODE = (1, 24, 8, 128, 8192, 40 * 1024 + 17, 9216)


def _attn(res, key, case, impl, seed, backward):
    lib = T.load()
    n, H, Hkv, hd, W, pos0, R = case
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn((n, H * hd), device="cuda", generator=g).to(torch.bfloat16)
    kr = torch.randn((Hkv, R, hd), device="cuda", generator=g).to(torch.bfloat16)
    vr = torch.randn((Hkv, R, hd), device="cuda", generator=g).to(torch.bfloat16)
    o = torch.zeros((n, H * hd), device="cuda", dtype=torch.bfloat16)
    lse = torch.zeros((H, n), device="cuda", dtype=torch.float32)
    rc = lib.ttt_kernel_attn_fwd(impl, n, H, Hkv, hd, W, R, pos0, q.data_ptr(), kr.data_ptr(), vr.data_ptr(),
                                 o.data_ptr(), lse.data_ptr(), n, None)
    assert rc == 0, (key, rc)
    res[key + "_o"] = o.float().cpu().numpy()
    res[key + "_lse"] = lse.cpu().numpy()
    if backward:
        dout = torch.randn((n, H * hd), device="cuda", generator=g).to(torch.bfloat16)
        dsum = torch.zeros((H, n), device="cuda", dtype=torch.float32)
        dqkv = torch.zeros((n, (H + 2 * Hkv) * hd), device="cuda", dtype=torch.bfloat16)
        rc = lib.ttt_kernel_attn_bwd(0, n, H, Hkv, hd, W, R, pos0, q.data_ptr(), kr.data_ptr(), vr.data_ptr(),
                                     o.data_ptr(), lse.data_ptr(), n, dout.data_ptr(), dsum.data_ptr(),
                                     dqkv.data_ptr(), None)
        assert rc == 0, (key, rc)
        res[key + "_dqkv"] = dqkv.float().cpu().numpy()
    torch.cuda.synchronize()
    assert T.ttt_kernel_error() == 0, key


def _context(res):
    # 3B widths, two blocks (one fast), chunks of 128, window 300: a prefill
    # of two chunks, then decode through a completed chunk into greedy picks
    s = inputs.shape("3b-4layer", n_layers=2, n_ttt_layers=1, chunk=128, window=300, seq_len=512)
    w, tok = inputs.make_weights(s), inputs.make_tokens(s)
    b = s.chunk
    P, N, n_given = 2 * b, b + 6, b - 10
    m = T.TTT(s, w, T.TTT_BF16, max_tokens=P + N + 1)
    try:
        res["ctx_prefill_losses"] = m.prefill(np.ascontiguousarray(tok[:P], np.int32))
        out, dl = m.decode(np.ascontiguousarray(tok[P:P + n_given], np.int32), N)
        res["ctx_decode_tokens"] = out
        res["ctx_decode_losses"] = dl
        fast = m.fast_weights(s.n_ttt_layers - 1)
        for k, v in fast.items():
            res["ctx_fast_" + k] = np.asarray(v, np.float32)
    finally:
        m.close()


def workload(out_path):
    res = {}
    for i, case in enumerate(ATTN):
        _attn(res, f"attn{i}", case, 0, 11 + i, backward=True)
    _attn(res, "decode", DECODE, 4, 21, backward=False)
    _context(res)
    count, kernel, index, limit = T.ttt_kernel_bounds()
    res["bounds"] = np.array([count, kernel, index, limit], np.int64)
    res["checked"] = np.array([int(T.ttt_kernel_bounds_checked())], np.int64)
    np.savez(out_path, **res)


def selftest():
    lib = T.load()
    assert lib.ttt_kernel_bounds_selftest(2, 3, None) == 0
    inside = T.ttt_kernel_bounds()
    assert lib.ttt_kernel_bounds_selftest(5, 3, None) == 0
    assert lib.ttt_kernel_bounds_selftest(-1, 3, None) == 0
    outside = T.ttt_kernel_bounds()
    after = T.ttt_kernel_bounds()
    print(json.dumps({"checked": T.ttt_kernel_bounds_checked(), "inside": inside, "outside": outside,
                      "after": after}))


if __name__ == "__main__":
    torch.cuda.set_device(0)
    if sys.argv[1] == "--selftest":
        selftest()
    else:
        workload(sys.argv[1])
