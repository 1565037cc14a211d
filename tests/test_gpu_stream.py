"""The bare-read reference (coli_moe_dbg_stream_read): one launch streams a
buffer through bulk copies and returns a checksum of it, which pins that every
byte range was copied (ragged tails, one and many blocks)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coli():
    import int4_routed_expert_f32_gb300 as c
    torch.cuda.set_device(0)
    return c


def _want(words: np.ndarray) -> int:
    # the four 32-bit words at every 1024-byte offset, summed modulo 2^64
    n = words.size * 4
    total = 0
    for o in range(0, n, 1024):
        total += int(words[o // 4: o // 4 + 4].astype(np.uint64).sum())
    return total % (1 << 64)


@pytest.mark.parametrize("n_bytes", [16, 1024, 16384 * 7 + 1040, 3 * (1 << 20) + 48, 64 * (1 << 20)])
def test_stream_read_checksum(coli, n_bytes):
    rng = np.random.default_rng(n_bytes)
    words = rng.integers(0, 1 << 32, size=n_bytes // 4, dtype=np.uint64).astype(np.uint32)
    buf = torch.from_numpy(words.view(np.int32).copy()).cuda()
    got = int(coli.dbg_stream_read(buf).cpu().numpy()[0]) % (1 << 64)
    assert got == _want(words)


@pytest.mark.parametrize("chunk,stages,bps", [(8192, 4, 2), (32768, 2, 3), (65536, 3, 1), (1024, 16, 4)])
def test_stream_read_ring_shapes(coli, chunk, stages, bps):
    """Other copy sizes, ring depths and blocks per SM read the same bytes."""
    n_bytes = 5 * (1 << 20) + 1024 + 32
    rng = np.random.default_rng(chunk + stages)
    words = rng.integers(0, 1 << 32, size=n_bytes // 4, dtype=np.uint64).astype(np.uint32)
    buf = torch.from_numpy(words.view(np.int32).copy()).cuda()
    got = coli.dbg_stream_read(buf, chunk=chunk, stages=stages, blocks_per_sm=bps)
    assert int(got.cpu().numpy()[0]) % (1 << 64) == _want(words)


def test_stream_read_prefix(coli):
    """n_bytes below the buffer's size reads only that prefix."""
    words = np.arange(1 << 16, dtype=np.uint32)
    buf = torch.from_numpy(words.view(np.int32).copy()).cuda()
    n = 5 * 1024 + 16
    got = int(coli.dbg_stream_read(buf, n_bytes=n).cpu().numpy()[0]) % (1 << 64)
    assert got == _want(words[: n // 4])
