"""The streaming-read measurement hook reads every byte it is given: the
sum it adds equals the sum of the buffer's 64-bit words modulo 2^64 computed
on the host, for empty, one-vector, ragged and multi-wave sizes."""

import numpy as np
import pytest
import torch

from speculative_decoding_verification_73_gb300 import binding, build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return binding.load()


@pytest.mark.parametrize("nbytes", [0, 16, 48 * 1024 + 16, 8 * 1024 * 1024 + 4096 + 48, 300 * 1024 * 1024])
def test_read_stream_checksum(nbytes):
    g = torch.Generator().manual_seed(nbytes % 9973)
    host = torch.randint(0, 256, (nbytes,), generator=g, dtype=torch.uint8)
    want = int(host.numpy().view(np.uint64).sum(dtype=np.uint64)) if nbytes else 0
    buf = host.cuda()
    got = binding.spec_verify_debug_read_stream(buf).item() & (2 ** 64 - 1)
    assert got == want
    # a second read adds to the same word
    out = torch.full((1,), 5, dtype=torch.int64, device="cuda")
    binding.spec_verify_debug_read_stream(buf, out)
    assert out.item() & (2 ** 64 - 1) == (want + 5) % 2 ** 64


def test_read_stream_refuses_ragged_sizes():
    buf = torch.zeros(40, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.SpecVerifyError):
        binding.spec_verify_debug_read_stream(buf)  # 40 bytes: not a multiple of 16
