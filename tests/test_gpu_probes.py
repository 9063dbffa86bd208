"""The peak probes the benchmark measures its roofline denominators with
(mttkrp_probe_fma, mttkrp_probe_mma): they run, finish within their bounded
wait, produce the arithmetic they claim, and reject bad arguments."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
import dense_tensor_decomposition_gb300 as mk  # noqa: E402

pytestmark = pytest.mark.gpu


def test_fma_probe_computes_its_chains():
    blocks, iters = 4, 100
    out = torch.zeros(blocks * 256, device="cuda")
    mk.probe_fma(blocks, iters, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    # each of the 8 chains: x <- x * m + b, iters times, from 1 + 1e-3 (c + (t & 7))
    t = np.arange(blocks * 256)
    want = np.zeros_like(got)
    m, b = np.float32(0.999999), np.float32(1e-7)
    for c in range(8):
        x = (np.float32(1.0) + np.float32(1e-3) * (c + (t & 7)).astype(np.float32)).astype(np.float32)
        for _ in range(iters):
            x = (x.astype(np.float64) * m + b).astype(np.float32)   # fma: one rounding
        want += x
    assert np.allclose(got, want, rtol=1e-6)


@pytest.mark.parametrize("kind", ["tf32", "f16"])
def test_mma_probe_runs_one_cta_per_sm(kind):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    mk.probe_mma(kind, sms, 256)
    torch.cuda.synchronize()
    assert mk.device_status() == 0


def test_probes_reject_bad_arguments():
    out = torch.zeros(256, device="cuda")
    with pytest.raises(mk.MttkrpError):
        mk.probe_fma(0, 10, out)
    with pytest.raises(KeyError):
        mk.probe_mma("bf8", 1, 1)
    lib = mk.load_library()
    assert lib.mttkrp_probe_mma(2, 1, 1, None) == 1
