"""The read-ceiling probe (a measurement aid of bench.py): it reads every
byte it is given, so the XOR of all 32-bit words it returns must equal the
host's, for any grid shape and for lengths that leave a ragged last pass."""
import numpy as np
import pytest

import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300.build import build_library

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("nwords", [0, 4, 4 * 1001, 1 << 20, (1 << 24) + 36])
@pytest.mark.parametrize("ctas,block", [(0, 0), (1, 1024), (4, 256), (8, 128), (-1, 0), (-1, 1024), (-1, 32)])
def test_probe_reads_every_word(nwords, ctas, block):
    rng = np.random.default_rng(nwords + block)
    w = rng.integers(0, 1 << 32, nwords, dtype=np.uint64).astype(np.uint32)
    x = torch.from_numpy(w.view(np.int32)).cuda()
    got = tcr.tcr_read_probe(x, ctas, block).cpu().numpy().view(np.uint32)[0]
    ref = np.bitwise_xor.reduce(w) if nwords else np.uint32(0)
    assert got == ref


def test_probe_rejects_bad_arguments():
    x = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(tcr.TcrError):
        tcr.tcr_read_probe(x[1:])            # not 16-byte aligned (and 252 bytes)
    with pytest.raises(tcr.TcrError):
        tcr.tcr_read_probe(x, 0, 48)         # block size not a power of two
