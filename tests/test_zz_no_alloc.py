"""The allocation-free decode entry point.

Some callers cannot allocate device memory while they run a decode step (a
plugin inside another inference runtime, a server whose memory planner reserved
all device memory at start-up), so they cannot hand the decode a workspace.
i8kv_int8_paged_decode_attn_noalloc runs the same kernel on a fixed scratch
array inside the library.  These checks call it through the C ABI and compare
it with the workspace entry point, on two calls in a row (the second call
reuses the scratch the first one left behind).  The file is named so that
pytest collects it last."""
import numpy as np
import pytest
import torch

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from tests.gpu_helpers import dev, host, gpu_decode_cache, gpu_quantize_rows, gpu_decode

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("lens,Hq,Hkv,D", [([5000, 1, 300, 0], 24, 4, 256), ([32768, 777], 32, 8, 128)])
def test_noalloc_matches_workspace_entry_point(lens, Hq, Hkv, D):
    w = wl.DecodeWorkload("noalloc", Hq, Hkv, D, lens, seed=12)
    cache = gpu_decode_cache(w)
    q_i8, q_s = gpu_quantize_rows(w.q(), w.Hkv, cache)
    ref = host(gpu_decode(w, cache, q_i8, q_s))
    bt, sl = dev(w.block_tables), dev(w.seq_lens)
    outs = [torch.full((w.B, Hq, D), float("nan"), dtype=torch.float32, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for call, out in enumerate(outs):
        i8.int8_paged_decode_attn_noalloc(out, q_i8, q_s, cache["k_cache"], cache["v_cache"], cache["k_scale"],
                                          cache["v_scale"], bt, sl)
        torch.cuda.synchronize()
        got = host(out)
        assert np.isfinite(got).all()
        # the same kernel with the same grid as the workspace entry point: the
        # same bits, on the first call and on the one after it (a stale or
        # aliased scratch would show here)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"call {call}"
        assert i8.device_error() == 0
    assert torch.cuda.mem_get_info()[0] == free_before  # the calls took no device memory


def test_noalloc_rejects_batches_beyond_the_fixed_scratch():
    B, Hq, Hkv, D = 4096, 24, 4, 256  # needs about (4096*4 + SMs) * 8256 bytes > 8 MiB
    out = torch.empty((1, 1), dtype=torch.float32, device="cuda")
    q_i8 = torch.zeros((B, Hq, D), dtype=torch.int8, device="cuda")
    q_s = torch.zeros((B, Hq), dtype=torch.float32, device="cuda")
    cache = i8.alloc_int8_cache(2, Hkv, D)
    bt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    sl = torch.ones((B,), dtype=torch.int32, device="cuda")
    with pytest.raises(i8.I8KVError) as e:
        i8.int8_paged_decode_attn_noalloc(out, q_i8, q_s, cache["k_cache"], cache["v_cache"], cache["k_scale"],
                                          cache["v_scale"], bt, sl)
    assert e.value.status == i8.binding.ERR_WORKSPACE and "scratch" in str(e.value)
