"""GPU parity of the layout kernels (pack, unpack, repack, validate, sym
detection) against the oracle: all bit-exact.  Calls go through the C ABI."""
import numpy as np
import pytest

import oracle
from oracle import oracle as npo
import bit_quantized_decode_unpack_gb300 as bqd
from bit_quantized_decode_unpack_gb300 import synth
from _util import to_dev

pytestmark = pytest.mark.gpu
F1, F2, T5 = bqd.FMT_AFFINE1, bqd.FMT_AFFINE2, bqd.FMT_T5


@pytest.mark.parametrize("fmt", [F1, F2, T5])
@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("N,K", [(1, 128), (3, 256), (17, 640), (130, 1280), (257, 5120)])
def test_pack_unpack_bit_exact(fmt, gs, N, K):
    import torch
    codes = synth.codes(np.random.default_rng(N * K + fmt + gs), fmt, N, K)
    w = bqd.pack(to_dev(codes), fmt, gs)
    back = bqd.unpack(w, N, K, fmt, gs)
    torch.cuda.synchronize()
    assert w.shape == (N, oracle.c_row_bytes(fmt, K, gs))
    assert np.array_equal(w.cpu().numpy(), oracle.c_pack(codes, fmt, gs))
    assert np.array_equal(back.cpu().numpy(), codes)


@pytest.mark.parametrize("fmt,N,K,gs", [(F1, 17408, 5120, 64), (F2, 5120, 17408, 128),
                                         (T5, 17408, 5120, 64), (T5, 5120, 17408, 128)])
def test_pack_full_size_bit_exact(fmt, N, K, gs):
    import torch
    codes = synth.codes(np.random.default_rng(5), fmt, N, K)
    w = bqd.pack(to_dev(codes), fmt, gs)
    torch.cuda.synchronize()
    assert np.array_equal(w.cpu().numpy(), oracle.c_pack(codes, fmt, gs))


@pytest.mark.parametrize("gs", [64, 128])
def test_unpack_every_t5_byte_value(gs):
    """Each of the 243 byte values, in non-final group positions, decodes to
    the oracle's trits."""
    import torch
    B = oracle.t5_bytes_per_group(gs)
    per_group = B - 1
    G = -(-243 // per_group)
    packed = np.zeros((1, G * B), dtype=np.uint8)
    vals = list(range(243))
    for g in range(G):
        for p in range(per_group):
            packed[0, g * B + p] = vals[(g * per_group + p) % 243]
    K = G * gs
    codes = bqd.unpack(to_dev(packed), 1, K, T5, gs)
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), oracle.c_unpack(packed, 1, K, T5, gs))


@pytest.mark.parametrize("gs", [64, 128])
def test_repack_2bit_to_t5(gs):
    import torch
    N, K = 33, 4 * gs
    codes = synth.codes(np.random.default_rng(gs), T5, N, K)  # ternary codes
    w2 = bqd.pack(to_dev(codes), F2, gs)
    w5, st = bqd.repack_2bit_to_t5(w2, N, K, gs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(w5.cpu().numpy(), oracle.c_pack(codes, T5, gs))
    bad = codes.copy()
    bad[0, 0] = 3
    bad[5, K - 1] = 3
    bad[32, 7] = 3
    w2b = bqd.pack(to_dev(bad), F2, gs)
    _, st = bqd.repack_2bit_to_t5(w2b, N, K, gs)
    assert int(st.item()) == 3


@pytest.mark.parametrize("gs", [64, 128])
def test_validate_t5_counts_match_oracle(gs):
    import torch
    N, K = 9, 3 * gs
    codes = synth.codes(np.random.default_rng(11), T5, N, K)
    packed = oracle.c_pack(codes, T5, gs)
    st = bqd.validate_t5(to_dev(packed), N, K, gs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    B = oracle.t5_bytes_per_group(gs)
    live = gs - 5 * (B - 1)
    bad = packed.copy()
    bad[0, 0] = 243
    bad[2, 2] = 255
    bad[4, B - 1] = 3 ** live
    bad[8, 3 * B - 1] = 200
    st = bqd.validate_t5(to_dev(bad), N, K, gs)
    assert int(st.item()) == oracle.c_t5_invalid_bytes(bad, N, K, gs) == 4
    # the counter is reset by each call
    st2 = bqd.validate_t5(to_dev(packed), N, K, gs, status=st)
    assert int(st2.item()) == 0


@pytest.mark.parametrize("ratio", [0.5, 1.5, 1.0, 0.3])
def test_detect_sym_matches_oracle(ratio):
    import torch
    rng = np.random.default_rng(3)
    s = synth.scales(rng, 300, 80)
    stored = npo.sym_bias(s, ratio)
    assert np.array_equal(oracle.c_sym_bias(s, ratio).view(np.uint16), stored.view(np.uint16))
    out = bqd.detect_sym(to_dev(s), to_dev(stored), ratio)
    torch.cuda.synchronize()
    assert int(out.item()) == 0
    changed = stored.copy()
    changed[1, 1] = -changed[1, 1]
    changed[299, 79] = np.float16(0)
    out = bqd.detect_sym(to_dev(s), to_dev(changed), ratio)
    assert int(out.item()) == oracle.c_sym_mismatches(s, changed, ratio) == 2
    asym = synth.biases(rng, F2, s)
    out = bqd.detect_sym(to_dev(s), to_dev(asym), ratio)
    assert int(out.item()) == oracle.c_sym_mismatches(s, asym, ratio)
