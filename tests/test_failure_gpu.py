"""Device-side failure path without a GPU fault: a bounded wait that nothing completes gives
up after its limit, the host reads OD_ERR_TIMEOUT with the wait's site word, the status is
cleared by the read, and the context keeps working."""
import pytest
import torch

from block_causal_video_attention_b300 import api, synth
from helpers import to_dev

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_context_survives():
    assert api.get_device_status() == 0
    api.selftest_expired_wait()
    st, site = api.get_device_status_detail()
    assert st == 4, api.STATUS.get(st, st)          # OD_ERR_TIMEOUT
    assert site >> 24 == 120 and site & 0x7FFFFF == 0   # the self-test's site, CTA 0
    assert api.get_device_status() == 0              # reading cleared it
    w = synth.WORKLOADS["tiny"]
    q, k, v = (to_dev(x) for x in synth.make_inputs(w, with_dout=False))
    o, lse = api.space_attn_fwd(q, k, v, w.agent, w.scale)
    torch.cuda.synchronize()
    assert api.get_device_status() == 0 and torch.isfinite(o.float()).all()
