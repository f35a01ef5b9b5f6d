"""Failure detection without a GPU fault: a kernel's bounded wait on a barrier
that nothing completes gives up after a short limit, the host reads
ATTNJVP_ETIMEOUT from the status word, attention launches skip their work
while the word is set, and after clearing it the context computes correctly."""
import time

import pytest
import torch

from attention_jvp_gb300 import binding, inputs
from helpers import assert_close, host64, oracle_on

pytestmark = pytest.mark.gpu


def _clear_status():
    try:
        binding.attn_jvp_status(clear=True)
    except binding.AttnJvpError:
        pass


def test_expired_wait_is_reported_and_context_stays_usable(cuda_lib):
    _clear_status()
    try:
        t0 = time.perf_counter()
        binding.attn_jvp_selftest_wait(20_000_000)  # 20 ms
        with pytest.raises(binding.AttnJvpError) as err:
            binding.attn_jvp_status(clear=False)
        elapsed = time.perf_counter() - t0
        assert err.value.code == binding.ATTNJVP_ETIMEOUT
        assert 0.02 <= elapsed < 10.0

        # While the word is set, attention kernels skip their work: outputs keep their sentinel.
        x = inputs.make_inputs(1, 2, 300, 128, seed=41, device="cuda")
        out = torch.full((1, 2, 300, 128), float("nan"), device="cuda")
        out_t = torch.full_like(out, float("nan"))
        binding.attn_jvp_fwd(x["q"], x["k"], x["v"], x["q_t"], x["k_t"], x["v_t"], scale=x["scale"],
                             out=out, out_t=out_t)
        torch.cuda.synchronize()
        assert bool(torch.isnan(out).all()) and bool(torch.isnan(out_t).all())
        with pytest.raises(binding.AttnJvpError):
            binding.attn_jvp_status(clear=True)  # still ETIMEOUT, now cleared

        # Cleared: the same launch now computes the right answer.
        got = binding.attn_jvp_fwd(x["q"], x["k"], x["v"], x["q_t"], x["k_t"], x["v_t"], scale=x["scale"],
                                   out=out, out_t=out_t)
        torch.cuda.synchronize()
        binding.attn_jvp_status()
        ref = oracle_on(x)
        assert_close(host64(got[0]).reshape(ref[0].shape), ref[0], "O")
        assert_close(host64(got[1]).reshape(ref[1].shape), ref[1], "Ot")
    finally:
        _clear_status()
