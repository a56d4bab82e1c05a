"""Pins of the encoder contract's operation order.

The pages fix the stages of the quantizer (Lynx reading, section 3) but not the
order of the fp32 operations inside them. The contract written for this build
(stated in include/lynx.h and in the oracle's header) fixes it: u = (x - mn) *
(1/rng), the chunk sum by the stride-halving tree over 32 slots, mean = sum /
n_c, and w = v * (1/s). Any other order is an equally plausible encoder that
produces different bytes, so each of these pages was chosen (by a search over
random chunks under the contract and under the alternative) so that the
alternative stores different metadata or codes. The expected bits below are
those the contract gives; the alternative's are noted beside them.

Every page holds channel 0 only (the other channels are zero): tokens 0 and 1
carry the page extremes 0.0 and 3.0, the other tokens of chunks 0..6 are 1.0,
and chunk 7 holds the crafted values (its first n_c tokens valid). With min 0
and range 3, u = x * fp32(1/3) (0x3EAAAAAB)."""
import numpy as np

BF16_1, BF16_3 = 0x3F80, 0x4040


def _page(chunk7):
    nc = len(chunk7)
    x = np.zeros((1, 1, 256, 128), np.uint16)
    x[0, 0, :224, 0] = BF16_1
    x[0, 0, 0, 0] = 0
    x[0, 0, 1, 0] = BF16_3
    x[0, 0, 224:224 + nc, 0] = np.asarray(chunk7, np.uint16)
    return x, np.array([224 + nc], np.int32)


def _chunk7(orc, chunk7):
    x, valid = _page(chunk7)
    q = orc.quantize(x, valid)
    nc = len(chunk7)
    pm = q["page_meta"][0, 0, 0, :, 0]
    assert pm[0] == 0.0 and pm[1] == 3.0
    mu, s = (int(v) for v in q["chunk_meta"][0, 0, 0, 7, :, 0])
    A = (q["anchor"][0, 0, 224:224 + nc, 0] & 15).astype(int)
    r = (q["residual"][0, 0, 224:224 + nc, 0] & 15).astype(int)
    codes = 16 * np.where(A >= 8, A - 16, A) + r - 7
    return mu, s, codes.tolist()


def test_u_is_a_product_with_the_reciprocal(orc):
    """32 equal values 2.21875 (bf16 0x400E): u = 2.21875 * fp32(1/3) is one
    fp32 ulp away from 2.21875 / 3, the mean is u itself and mu = fp16(u) =
    0x39EB; the scale s = fp16 up(|u - mu|) is 0x0955 under the contract and
    0x0956 with a division."""
    mu, s, codes = _chunk7(orc, [0x400E] * 32)
    assert (mu, s) == (0x39EB, 0x0955)
    assert codes == [-63] * 32


SEQ_CHUNK = [0x3FF6, 0x3FE0, 0x3FDF, 0x3FFA, 0x3FFA, 0x3FDF, 0x3FDF, 0x3FE2, 0x3FD9, 0x3FEF, 0x3FF5, 0x3FF9,
             0x3FF1, 0x3FF7, 0x3FE0, 0x3FF7, 0x3FD9, 0x3FF7, 0x3FF7, 0x3FDB, 0x3FE1, 0x3FE0, 0x3FE2, 0x3FED,
             0x3FEE, 0x3FE2, 0x3FE4, 0x3FE6, 0x3FF9, 0x3FFD, 0x3FE8, 0x3FF3]


def test_chunk_sum_is_the_stride_halving_tree(orc):
    """A chunk of values near 1.8: the tree sum's mean rounds to mu = 0x38E4 and
    gives s = 0x2A16; a left-to-right sum gives mu = 0x38E5, s = 0x2A06, and
    codes that differ at tokens 0, 9, 19, 23, 24 and 30."""
    mu, s, codes = _chunk7(orc, SEQ_CHUNK)
    assert (mu, s) == (0x38E4, 0x2A16)
    assert codes == [58, -57, -58, 61, 61, -58, -58, -55, -63, 47, 56, 60, 51, 58, -57, 58, -63, 58, 58, -61, -56,
                     -57, -55, 40, 44, -55, -52, -48, 60, 63, -42, 54]


W_CHUNK = [0x3FC4, 0x4002, 0x3FEE, 0x3FDD, 0x3F9D, 0x400B, 0x3FD9, 0x3F93, 0x3FFC, 0x3FAE, 0x3FB3, 0x3FFF,
           0x400F, 0x3F9E, 0x3FB4, 0x3F93, 0x3F9D, 0x3FB0, 0x4006, 0x3FA8, 0x4010, 0x3FD5, 0x3FE1, 0x3FC4,
           0x3FCD, 0x3F93, 0x3FC3, 0x3FD8, 0x3F97, 0x400D, 0x3FB7, 0x3FFA]


def test_w_is_a_product_with_the_reciprocal(orc):
    """mu = 0x3857, s = 0x32A4 either way; token 21's w = v * fp32(1/s) falls
    below threshold T_32 (code 31) where v / s reaches it (code 32)."""
    mu, s, codes = _chunk7(orc, W_CHUNK)
    assert (mu, s) == (0x3857, 0x32A4)
    assert codes == [-42, 58, 52, 42, -58, 61, 38, -60, 56, -53, -52, 57, 63, -58, -51, -60, -58, -53, 60, -55, 63,
                     31, 45, -42, -28, -60, -43, 37, -59, 62, -50, 56]


def test_mean_is_a_division_by_the_valid_count(orc):
    """A ragged chunk of 7 valid tokens: sum / 7 rounds to mu = 0x2DD4 (then
    s = 0x308C); sum * fp32(1/7) rounds to 0x2DD5 (s = 0x308B)."""
    mu, s, codes = _chunk7(orc, [0x3D7F, 0x3D9E, 0x3F2B, 0x3B85, 0x3ECE, 0x0000, 0x3F33])
    assert (mu, s) == (0x2DD4, 0x308C)
    assert codes == [-55, -54, 62, -58, 50, -58, 63]
