"""RoPE tables (RoPE article, section 2.2 and footnote 3): the CUDA table against the
float64 oracle's angles, entry by entry.

Each entry holds cos and sin of pos * theta^(-2j/d) as a pair of fp32 parts: hi with
at most 16 significant bits (so that a bf16 times hi is exact in fp32) and lo, the
fp32 rounding of the remainder.  hi + lo must equal the fp64 value to within the
rounding of the fp64 angle itself (|angle| * 2^-52) plus lo's fp32 rounding."""

import numpy as np
import pytest
import torch

import oracle.pic_oracle as O
import position_independent_kv_pic_gb300 as pic
from position_independent_kv_pic_gb300 import build as pic_build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pic_build.build()
    pic.load()


def _table(pos, d, theta):
    p = torch.tensor(pos, dtype=torch.int32, device="cuda")
    t = torch.empty((len(pos), d // 2, 4), dtype=torch.float32, device="cuda")
    pic.pic_rope_table(p, d, theta, t)
    torch.cuda.synchronize()
    return t.double().cpu().numpy()


def _bits_used(x):
    """Significant bits of each fp32 value (0 for zero)."""
    m = np.frexp(np.abs(x.astype(np.float64)))[0] * 2.0 ** 24
    m = m.astype(np.int64)
    tz = np.zeros_like(m)
    nz = m != 0
    mm = m[nz]
    tz[nz] = np.log2(mm & -mm).astype(np.int64)
    return np.where(nz, 24 - tz, 0)


@pytest.mark.parametrize("d,theta", [(128, 5e5), (128, 1e4), (64, 1e4), (2, 1e4), (256, 1e6)])
def test_table_matches_fp64_angles(d, theta):
    rng = np.random.default_rng(d + int(theta) % 97)
    pos = np.concatenate([[0, 1, 2, 15, 16, 1000, 100_255, 2**20, 2**24 - 1],
                          rng.integers(0, 2**21, size=700)]).astype(np.int64)
    tab = _table(pos.tolist(), d, theta)
    ang = pos[:, None].astype(np.float64) * O.inv_freq(d, theta)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    bound = np.abs(ang) * 2.0 ** -52 + 2.0 ** -40
    assert np.all(np.abs(tab[..., 0] + tab[..., 2] - c) <= bound)
    assert np.all(np.abs(tab[..., 1] + tab[..., 3] - s) <= bound)
    # hi carries at most 16 significant bits; lo is below hi's last bit
    assert _bits_used(tab[..., 0]).max() <= 16 and _bits_used(tab[..., 1]).max() <= 16
    assert np.all(np.abs(tab[..., 2]) <= np.abs(tab[..., 0]) * 2.0 ** -15 + 2.0 ** -40)
    # position 0 is the identity rotation
    assert np.all(tab[0, :, 0] == 1.0) and np.all(tab[0, :, 1:] == 0.0)


def test_table_size_not_a_multiple_of_the_block():
    """A table whose entry count is not a multiple of the block size and spans more
    blocks than the grid holds (grid-stride tail)."""
    d, theta = 128, 5e5
    n = 152 * 32 * 64 // (d // 2) * 3 + 5
    pos = (np.arange(n, dtype=np.int64) * 7919) % 300_000
    tab = _table(pos.tolist(), d, theta)
    ang = pos[:, None].astype(np.float64) * O.inv_freq(d, theta)[None, :]
    bound = np.abs(ang) * 2.0 ** -52 + 2.0 ** -40
    assert np.all(np.abs(tab[..., 0] + tab[..., 2] - np.cos(ang)) <= bound)
    assert np.all(np.abs(tab[..., 1] + tab[..., 3] - np.sin(ang)) <= bound)
