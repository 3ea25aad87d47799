"""The decoder's bounded device waits: a wait that runs out reports
CG_ERR_TIMEOUT instead of spinning, leaves nothing in flight, and the context
stays usable.  The wait is made to run out by the library's test kernel
(cg_test_decode_timeout), which never requests one ring segment of each
stream and polls only briefly; nothing faults or hangs the GPU."""
import time

import numpy as np
import pytest
import torch

from oracle import oracle as O
from kv_cache_compression_decode_gb300 import codec as C
from kv_cache_compression_decode_gb300 import synth
from tests import parity as P

pytestmark = pytest.mark.gpu
needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")

WAIT_BIT = 1 << 22  # diagnostic bit: a bounded device wait gave up


@needs_gpu
@pytest.mark.parametrize("source", ["gpu-encoded", "oracle-encoded"])
def test_bounded_wait_runs_out_reports_timeout_and_context_survives(source):
    L, T, Cc, tps = 4, 700, 256, 256
    x = synth.ar1_kv(L, T, Cc, 0.95, 2, seed=21)
    pc, oc = P.configs(L, T, Cc, 10, 0, tps)
    oenc = O.encode(oc, x.numpy().view(np.uint16))
    expect = O.decode(oc, oenc)
    enc = C.encode(pc, x.cuda()) if source == "gpu-encoded" else P.upload(oenc)
    sizes = np.diff(oenc.stream_off.astype(np.int64))
    assert (sizes > 256).all()  # every stream needs the withheld segment

    out = torch.full((L, 2, T, Cc), float("nan"), dtype=torch.float16, device="cuda")
    st = C.new_status()
    t0 = time.perf_counter()
    C.cg_test_decode_timeout(pc, enc, out, st)
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    flags = int(st.item()) & 0xFFFFFFFF
    assert flags == (1 << C.CG_ERR_TIMEOUT) | WAIT_BIT, hex(flags)
    assert C.read_status(st) == C.CG_ERR_TIMEOUT
    assert took < 5.0  # every wait is bounded: the kernel returned on its own

    # the same object, destination and context decode normally afterwards
    for _ in range(2):
        st = C.new_status()
        C.cg_decode(pc, enc, out, st)
        torch.cuda.synchronize()
        assert C.read_status(st) == C.CG_OK
        assert np.array_equal(out.cpu().numpy().view(np.uint16), expect)
