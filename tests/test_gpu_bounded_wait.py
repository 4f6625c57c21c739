"""The attention's failure path on the GPU, without a fault.  A packed split
waits for each staged tile with a bounded mbarrier wait, and an overlapping
call waits for the previous call's epoch with a bounded wait; here the same
waits run on a barrier phase that nothing completes and on an epoch that
nothing publishes.  Each must give up after its 200 ms limit, report through
the status word the host reads (bits 1 and 2), and leave the context usable:
an attention launched right after still matches the oracle."""
import time

import numpy as np
import pytest
import torch

from bit_kv_cache_kivi_gb300 import workloads as W
import kivi_testlib as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from bit_kv_cache_kivi_gb300 import build, kivi
    build.build()
    kivi.lib()
    torch.cuda.init()


def test_bounded_wait_gives_up_and_reports():
    from bit_kv_cache_kivi_gb300 import kivi as K
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    K.kivi_check_bounded_wait(st)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert st.item() == 3
    assert 0.38 < dt < 10.0, dt

    # the context is intact: a prefill and an attention right after
    wl = W.synthetic("bw", B=2, Hq=8, Hkv=2, T=300, R=32, seed=3)
    g = T.gpu_cache(wl, capacity=320)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    o = T.oracle_cache(wl, capacity=320)
    o.prefill(wl.k, wl.v)
    out = T.out_float(g.attention(T.dev(wl.q, wl.q_dtype)))
    assert T.attn_err(out, o.attention(T.q_float(wl.q, wl.q_dtype))) <= T.ATTN_TOL


def test_bounded_wait_status_pointer_checks():
    from bit_kv_cache_kivi_gb300 import kivi as K
    page = np.zeros(4, np.int32)  # pageable host memory: not reachable by the kernel
    assert K.lib().kivi_check_bounded_wait(page.ctypes.data, None) == K.KIVI_EINVAL
    with pytest.raises(K.KiviError):
        K.kivi_check_bounded_wait(torch.zeros(1, dtype=torch.float32, device="cuda"))
