"""Race detector for the decode kernel: with identical inputs the kernel is
deterministic (fixed work split, fixed merge order), so repeated launches must
give bit-identical outputs.  A producer/consumer or cross-CTA merge race shows
up as a run that differs.  Runs the FP8 and NVFP4 variants on a 44-sequence
batch whose (sequence, head) pairs are split across CTAs, with the allocator
state disturbed between runs."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("prec", [0, 1])
def test_repeated_decodes_are_bit_identical(prec):
    from nvfp4_quantized_paged_gb300.runner import Layer
    from nvfp4_quantized_paged_gb300.workloads import SPECS, Workload, scaled
    spec = scaled(SPECS["mixed28_b44"], layers=1, fp8_layers=())
    wl = Workload(spec, seed=1, device="cuda")
    lay = Layer(wl, 0, prec=prec)
    lay.decode()
    ref = lay.out.clone()
    for it in range(12):
        junk = torch.empty(int(3e8) + it * 4096, dtype=torch.uint8, device="cuda").fill_(0xFF)
        lay.out.fill_(0)
        lay.decode()
        del junk
        assert torch.equal(lay.out, ref), f"run {it} differs"
        assert lay.cache.err.item() == 0


@pytest.mark.parametrize("prec", [0, 1])
def test_repeated_weighted_share_decodes_are_bit_identical(prec):
    """The same check on a 256-sequence batch of log-normal lengths: 2048
    (sequence, KV head) pairs for the CTAs, so the launch weighs shares by
    pairs and most CTAs cut two pairs."""
    from nvfp4_quantized_paged_gb300.runner import Layer
    from nvfp4_quantized_paged_gb300.workloads import SPECS, Workload, scaled
    spec = scaled(SPECS["serving_mix_b256"], extend_seqs=(), extend_tokens=0)
    wl = Workload(spec, seed=2, device="cuda")
    lay = Layer(wl, 0, prec=prec)
    lay.decode()
    ref = lay.out.clone()
    for it in range(6):
        lay.out.fill_(0)
        lay.decode()
        assert torch.equal(lay.out, ref), f"run {it} differs"
        assert lay.cache.err.item() == 0
