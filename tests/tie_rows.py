"""fp16 activation rows that land the int8 activation codes on exact ties.

Test input construction only (it uses scipy's Hadamard matrix). The rows are
x = H.S / 128 for chosen integer Hadamard-domain sums S. Every such x is exact
in fp16 (multiples of 1/128 below 16), and the binary32 butterflies of the
input transform reproduce S exactly. Every row has S = 508 at position 0
(its absmax) and three entries S = +-2s with s odd, for which
127 * S / 508 = s / 2 lies exactly halfway between two integer codes.
"""
import numpy as np
import scipy.linalg

_H = scipy.linalg.hadamard(128).astype(np.int64)


def tie_rows():
    """(x fp16 [43][128], suh fp16 ones [128], S int64 [43][128])."""
    rows, sums = [], []
    odd = list(range(1, 254, 2))
    for i in range(0, len(odd), 3):
        S = np.zeros(128, np.int64)
        S[0] = 508
        for j, s in enumerate(odd[i:i + 3]):
            S[1 + 5 * j + i % 7] = 2 * s * (-1 if (i + j) % 2 else 1)
        v = _H @ S
        assert np.abs(v).max() < 2048
        rows.append(v / 128.0)
        sums.append(S)
    x = np.array(rows, dtype=np.float16)
    assert np.array_equal(x.astype(np.float64), np.array(rows))
    return x, np.ones(128, np.float16), np.array(sums)
