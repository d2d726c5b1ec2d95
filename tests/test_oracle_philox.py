"""Pin the oracle's Philox4x64-10 against numpy's independent implementation.

numpy.random.Philox is Philox4x64-10 (Salmon et al., SC'11).  It advances its
counter by one *before* producing each block of four words, so the block for
counter c is the first output of a generator whose counter is set to c - 1.
"""
import numpy as np
import pytest

import oracle

M64 = (1 << 64) - 1


def numpy_block(ctr, key):
    words = list(ctr)
    # counter - 1 with borrow across the four 64-bit words
    i = 0
    while True:
        if words[i] == 0:
            words[i] = M64
            i += 1
            if i == 4:
                break
        else:
            words[i] -= 1
            break
    bg = np.random.Philox(counter=np.array(words, np.uint64), key=np.array(key, np.uint64))
    return bg.random_raw(4).astype(np.uint64)


CASES = [
    ((0, 0, 0, 0), (0, 0)),
    ((M64, M64, M64, M64), (M64, M64)),
    ((1, 0, 0, 0), (0, 0)),
    ((0, 1, 0, 0), (7, 0)),
    ((255, 16, 0, 0), (12345, 0)),
    ((0x243F6A8885A308D3, 0x13198A2E03707344, 0xA4093822299F31D0, 0x082EFA98EC4E6C89),
     (0x452821E638D01377, 0xBE5466CF34E90C6C)),
]


@pytest.mark.parametrize("ctr,key", CASES)
def test_philox_matches_numpy(ctr, key):
    got = oracle.philox4x64_10(np.array(ctr, np.uint64), np.array(key, np.uint64))
    want = numpy_block(ctr, key)
    assert [int(x) for x in got] == [int(x) for x in want]


def test_philox_random_counters_match_numpy():
    rng = np.random.default_rng(5)
    for _ in range(64):
        ctr = [int(x) for x in rng.integers(0, 2**63, 4, dtype=np.int64)]
        key = [int(x) for x in rng.integers(0, 2**63, 2, dtype=np.int64)]
        got = oracle.philox4x64_10(np.array(ctr, np.uint64), np.array(key, np.uint64))
        assert [int(x) for x in got] == [int(x) for x in numpy_block(ctr, key)]


def test_uniforms_are_top_24_bits_of_words_0_1_2():
    for seed, b, k in [(0, 0, 0), (0, 3, 8), (17, 255, 16), (2**40 + 3, 1, 2)]:
        us = oracle.uniforms(seed, b, k)
        block = numpy_block((b, k, 0, 0), (seed, 0))
        for w, u in zip(block[:3], us):
            assert u == int(w >> np.uint64(40)) / 2.0**24
            assert 0.0 <= u < 1.0
            assert float(np.float32(u)) == u        # exact in fp32


def test_uniforms_are_uniform():
    from scipy import stats
    us = np.array([oracle.uniforms(3, b, k)[0] for b in range(400) for k in range(17)])
    assert stats.kstest(us, "uniform").pvalue > 1e-3
