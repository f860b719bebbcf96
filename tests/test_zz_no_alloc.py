"""gdn_chunk_fwd_noalloc: the two-pass chunk forward with the library's static scratch.

Collected last (file name), and independent of every other test file: it passes
alone and after the rest.  The GPU tests check two consecutive calls against the
caller-workspace entry point bit for bit; the CPU test checks that a request
above the 64 MiB scratch is refused before anything is launched.
"""
import ctypes

import numpy as np
import pytest
import torch

import gated_delta_rule_gdn_gb300 as gdn
from gated_delta_rule_gdn_gb300 import _binding, build, workloads as W

SCRATCH_BYTES = 64 << 20
ITEM_BYTES = 74240


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gdn.load()


def test_oversized_request_is_refused_before_any_launch(lib):
    fake = 0x10000
    B, T, H = 4, 4096, 16          # (256 + 4 + 1) * 16 items of 74,240 bytes > 64 MiB
    assert (B * T // 64 + B + 1) * H * ITEM_BYTES > SCRATCH_BYTES
    st = lib.gdn_chunk_fwd_noalloc(0, fake, fake, fake, fake, fake, 0.1, None, 0, None, None, 0, fake,
                                   B, T, H, 128, 128, 64, 1, 0, None)
    assert st == 2
    msg = _binding.last_error()
    assert "scratch" in msg and str(SCRATCH_BYTES) in msg


def _inputs(kind, seed, T, H):
    cfg = W.config(3 if kind == "kda" else 1)
    x = W.chunk_inputs(cfg, seed=seed, B=1, T=T, H=H)
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}, kind == "kda"


def _ref(x, per_channel):
    fn = gdn.kda_chunk_fwd if per_channel else gdn.gdn_chunk_fwd
    o, h = fn(x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"], initial_state=x["initial_state"],
              output_final_state=True, algo="two_pass")
    return o, h


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_two_consecutive_calls_match_the_workspace_entry_point(lib, kind):
    T, H = 1000, 4                  # (15 + 1 + 1) * 4 items: well inside the scratch
    xa, pc = _inputs(kind, 11, T, H)
    xb, _ = _inputs(kind, 12, T, H)
    outs = []
    for x in (xa, xb):              # the second call reuses the scratch the first one wrote
        o, h = gdn.chunk_fwd_noalloc(pc, x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"],
                                     initial_state=x["initial_state"], output_final_state=True)
        outs.append((o, h))
    torch.cuda.synchronize()
    assert gdn.device_status() == 0
    for (o, h), x in zip(outs, (xa, xb)):
        o_ref, h_ref = _ref(x, pc)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref)
        assert torch.equal(h, h_ref)
    assert not torch.equal(outs[0][0], outs[1][0])


@pytest.mark.gpu
def test_largest_request_that_fits(lib):
    H = 12
    T = 4096                        # (64 + 2) * 12 = 792 items, 65.3 MB <= 64 MiB
    assert (T // 64 + 2) * H * ITEM_BYTES <= SCRATCH_BYTES
    x, pc = _inputs("gdn", 13, T, H)
    o, h = gdn.chunk_fwd_noalloc(pc, x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"],
                                 initial_state=x["initial_state"], output_final_state=True)
    o_ref, h_ref = _ref(x, pc)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(h, h_ref)
