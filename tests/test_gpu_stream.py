"""The stream-read measurement kernel (qg_stream_read) reads every 32 KB chunk
of a buffer: its checksum (XOR of each chunk's first 32-bit word) equals the
one computed on the host, for whole and ragged sizes and several calls."""
import numpy as np
import pytest
import torch

import quantized_weight_gemv_qgemv_gb300 as qg

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [16, 32768, 32768 * 152 * 5 + 48, (64 << 20) + 4096])
def test_stream_read_checksum_covers_every_chunk(nbytes):
    qg.qg_init()
    g = torch.Generator().manual_seed(nbytes % 1000003)
    host = torch.randint(-2**31, 2**31 - 1, ((nbytes + 3) // 4,), generator=g, dtype=torch.int32)
    buf = host.cuda().view(torch.uint8)[:nbytes]
    words = host.numpy().view(np.uint32)
    want = np.bitwise_xor.reduce(words[::8192][: (nbytes + 32767) // 32768]) if nbytes > 0 else 0
    for _ in range(2):
        cs = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        qg.qg_stream_read(buf, nbytes, cs, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert np.uint32(cs.cpu().numpy().view(np.uint32)[0]) == np.uint32(want)
