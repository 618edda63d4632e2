"""Host-side checks of the Python layer (no GPU): argument validation of the mixer helpers and
the gate-mode flags' values against include/kda.h."""

import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mods():
    from gated_delta_rule_scan_gb300 import _build
    _build.build()
    from gated_delta_rule_scan_gb300 import kda, mixer
    return kda, mixer


def test_flag_values_match_header(mods):
    kda, _ = mods
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    defs = dict(re.findall(r"#define (KDA_\w+) (\d+)", text))
    assert int(defs["KDA_GATE_PER_CHANNEL"]) == kda.GATE_PER_CHANNEL
    assert int(defs["KDA_GATE_PER_HEAD"]) == kda.GATE_PER_HEAD
    assert int(defs["KDA_GATE_EXP"]) == kda.GATE_EXP
    assert int(defs["KDA_NORM_SILU"]) == kda.NORM_SILU
    # the flags are distinct bits
    assert kda.GATE_PER_HEAD & kda.GATE_EXP == 0 and kda.NORM_SILU & (kda.GATE_PER_HEAD | kda.GATE_EXP) == 0


def test_norm_gate_names(mods):
    _, mixer = mods
    assert mixer._norm_flag("sigmoid") == 0
    assert mixer._norm_flag("silu") != 0
    with pytest.raises(ValueError):
        mixer._norm_flag("relu")


def test_host_stream_needs_device_weights(mods):
    _, mixer = mods
    w = torch.zeros(4)
    with pytest.raises(ValueError):
        mixer.HostPrefillStream(like={}, conv_w=None, dt_bias=w, a_log=w, norm_w=w, H=1, N=1, T=1)
