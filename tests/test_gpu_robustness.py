"""Bounded device waits: a wait that nothing satisfies gives up, records
SAGE_ERR_TIMEOUT in the workspace status word and leaves the context usable."""
import pytest
import torch

import bit_trainable_attention_sagebwd_gb300 as sa

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    ws = sa.alloc_ws(1, 1, 128, 64)
    ws.zero_()
    s = sa._stream_ptr()
    assert sa.sage_attn_selftest_wait(sa._ptr(ws), 1_000_000, s) == sa.SAGE_OK  # 1 ms budget
    assert sa.get_status(ws) == sa.SAGE_ERR_TIMEOUT
    assert sa.get_status(ws) == sa.SAGE_OK  # read clears the word
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0  # the context still works


def test_unsupported_shapes_raise():
    q = torch.zeros(1, 1, 128, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sa.SageError):
        sa.quantize(q, q, q)
