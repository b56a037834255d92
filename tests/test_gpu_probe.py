"""The measurement kernels run to completion and leave no error: the FP8
MMA-rate kernel in both shapes (one CTA, and CTA pairs issuing cta_group::2
MMAs) and the TMEM read-rate kernel in both load patterns."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nfq():
    import norm_fp8_quant_gb300 as m
    from norm_fp8_quant_gb300 import build
    build.build()
    m.load()
    assert torch.cuda.is_available()
    return m


@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("stages", [1, 4])
def test_probe_fp8_mma_runs(nfq, pair, stages):
    flops = nfq.probe_fp8_mma(pair, 4, 16, stages)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    assert flops == 2.0 * (256 if pair else 128) * 256 * 128 * 16 * 4
    with pytest.raises(nfq.NfqError):
        nfq.probe_fp8_mma(pair, 0, 16)
    with pytest.raises(nfq.NfqError):
        nfq.probe_fp8_mma(pair, 4, 16, 5)


@pytest.mark.parametrize("pair", [False, True])
def test_probe_nvfp4_mma_runs(nfq, pair):
    flops = nfq.probe_nvfp4_mma(pair, 4, 16)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    assert flops == 2.0 * (256 if pair else 128) * 256 * 256 * 16 * 4
    with pytest.raises(nfq.NfqError):
        nfq.probe_nvfp4_mma(pair, 0, 16)


@pytest.mark.parametrize("m,n", [(128, 256), (128, 16), (64, 256), (64, 8 * 3 + 16)])
def test_probe_fp8_mma_shape_runs(nfq, m, n):
    assert nfq.probe_fp8_mma_shape(m, n, 4, 16) == 2.0 * m * n * 128 * 16 * 4
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    with pytest.raises(nfq.NfqError):
        nfq.probe_fp8_mma_shape(128, 24, 4, 16)      # N not a multiple of 16 for M = 128


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_probe_handoff_runs(nfq, mode):
    assert nfq.probe_handoff(mode, 64) == 128
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    with pytest.raises(nfq.NfqError):
        nfq.probe_handoff(4, 64)


def test_probe_mma_with_tmem_readers_runs(nfq):
    flops = nfq.probe_fp8_mma(False, 4, 64, 0)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    assert flops == 2.0 * 128 * 256 * 128 * 64 * 4
    with pytest.raises(nfq.NfqError):
        nfq.probe_fp8_mma(True, 4, 16, 0)


@pytest.mark.parametrize("batched", [False, True])
def test_probe_tmem_ld_runs(nfq, batched):
    nbytes = nfq.probe_tmem_ld(batched, 4, 8)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    assert nbytes == 128.0 * 256 * 4 * 8 * 4


@pytest.mark.parametrize("T,H,k", [(64, 6144, 8), (1, 7168, 8), (700, 1024, 3)])
def test_probe_stage1_reads_runs(nfq, T, H, k):
    parts = [torch.randn(T, H, device="cuda").to(torch.bfloat16) for _ in range(k)]
    res = torch.randn(T, H, device="cuda").to(torch.bfloat16)
    nfq.prepare_probe_stage1_reads(parts, res)()
    torch.cuda.synchronize()
    assert nfq.device_error() == 0


@pytest.mark.parametrize("pair,buffers,mode",
                         [(p, b, m) for p, b in ((False, 2), (False, 4), (False, 8), (True, 2),
                                                 (True, 4)) for m in (0, 1, 2)]
                         + [(False, 4, 3), (True, 4, 3)])
def test_probe_handshake_runs(nfq, pair, buffers, mode):
    """The accumulator hand-off probe runs every K block through its buffers and
    leaves no expired wait, with and without an epilogue."""
    assert nfq.probe_handshake(pair, buffers, mode, 4, 64) == 64
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    with pytest.raises(nfq.NfqError):
        nfq.probe_handshake(pair, 6, mode, 4, 64)


def test_expired_wait_sets_the_error_word_and_the_context_stays_usable(nfq):
    """Failure detection without a fault: a kernel's bounded wait on a barrier
    nothing arrives on gives up after its limit, the host reads
    NFQ_ERR_TIMEOUT from the device error word (cleared by the read), and the
    next launches run normally on the same context."""
    import time
    assert nfq.device_error() == nfq.NFQ_OK
    t0 = time.time()
    nfq.probe_wait_timeout()
    assert nfq.device_error() == nfq.NFQ_ERR_TIMEOUT
    waited = time.time() - t0
    assert 1.5 < waited < 30.0, waited
    assert nfq.device_error() == nfq.NFQ_OK           # the read cleared it
    # the context still runs tensor-core work afterwards and leaves no error
    assert nfq.probe_fp8_mma(False, 4, 16) > 0
    torch.cuda.synchronize()
    assert nfq.device_error() == nfq.NFQ_OK
