"""GPU parity of INT8 decode with UINT8 probability codes (0..255, sW = A / 255,
the s8 x u8 MMA) against the oracle run with the same code range, on the same
seeded inputs; same 2e-3 max-abs bar as the signed-code decode.  Also checks
that the extra bit shows: against fp64 attention on the dequantized cache the
UINT8 variant's error is clearly below the signed variant's."""
import numpy as np
import pytest

import int8_kv_cache_token_gb300 as i8
import workloads as wl
from oracle import oracle as orc
from tests.gpu_helpers import host, gpu_decode_cache, gpu_quantize_rows, gpu_decode
from tests.helpers import oracle_decode_cache, oracle_query, gather_int8

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.mark.parametrize("D,Hq,Hkv,lens", [(256, 24, 4, [4096]), (128, 32, 8, [513, 1, 2000, 77]),
                                             (256, 8, 1, [300, 9000])])
def test_decode_u8_probs_matches_oracle(D, Hq, Hkv, lens):
    w = wl.DecodeWorkload("u8p", Hq, Hkv, D, lens, seed=len(lens) + D)
    cache = gpu_decode_cache(w)
    q_i8, q_s = gpu_quantize_rows(w.q(), Hkv, cache)
    out = host(gpu_decode(w, cache, q_i8, q_s, u8_probs=True))
    assert i8.device_error() == 0
    oc = oracle_decode_cache(w)
    oq, oqs = oracle_query(w)
    ref = orc.decode_attn(oq, oqs, oc, w.block_tables, w.seq_lens, w.block_size, pmax=255)
    err = np.abs(out - ref).max()
    assert err <= TOL, f"max-abs {err:.3e}"


def test_decode_u8_probs_halves_probability_error():
    # the outlier workload at 8192: error of each variant against fp64 softmax
    # attention over the same dequantized cache (only the probability codes differ)
    w = wl.decode_outlier(8192)
    cache = gpu_decode_cache(w)
    q_i8, q_s = gpu_quantize_rows(w.q(), w.Hkv, cache)
    s8 = host(gpu_decode(w, cache, q_i8, q_s))
    u8 = host(gpu_decode(w, cache, q_i8, q_s, u8_probs=True))
    oc = oracle_decode_cache(w)
    L, D, G = 8192, w.D, w.Hq // w.Hkv
    Kt, Vt, sK, sV = gather_int8(oc, w.block_tables[0], L, w.Hkv, D)
    qi, qs = host(q_i8), host(q_s)
    c = float(np.float32(1) / np.sqrt(np.float32(D)))
    e8, e16 = [], []
    for h in range(w.Hq):
        kv = h // G
        s = (Kt[:, kv].astype(np.int64) @ qi[0, h].astype(np.int64)) * float(qs[0, h]) * sK[:, kv] * c
        p = np.exp(s - s.max())
        ref = (p / p.sum()) @ (Vt[:, kv] * sV[:, kv, None].astype(np.float64))
        e8.append(np.abs(s8[0, h] - ref).mean())
        e16.append(np.abs(u8[0, h] - ref).mean())
    assert np.mean(e16) < 0.7 * np.mean(e8), (np.mean(e16), np.mean(e8))
