"""Chunk planner: the wave rules of the instruction-bound passes ("Flash
Decoding" tutorial, section 3: split the keys so that the whole GPU is busy;
its "common misconceptions" section: more chunks are not free).

The fp4 pass runs 3 CTAs per SM and the fused top-delta pass 2 (their
occupancy on sm_103a); both are limited by their SM's instruction issue, so
the planner fills every resident slot in one wave where the shape allows and
charges each further wave a fixed cost.  These tests pin the chunk counts the
planner returns through the C ABI on the device's own SM count.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

FP4_CTAS_PER_SM = 3
TOPDELTA_CTAS_PER_SM = 2


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("B,Hq,Hkv,L", [(1, 32, 8, 1 << 20), (4, 32, 8, 131072), (1, 32, 32, 32768)])
def test_fp4_plan_fills_one_wave(fd, B, Hq, Hkv, L):
    slots = FP4_CTAS_PER_SM * _sms()
    S = fd.fd_num_splits_fp4(B, Hq, Hkv, L, 128)
    ctas = B * Hkv * S
    assert ctas <= slots, (S, ctas, slots)               # one wave
    assert ctas + B * Hkv > slots, (S, ctas, slots)      # no further chunk fits in it


def test_fp4_plan_explicit_count_wins(fd):
    assert fd.fd_num_splits_fp4(1, 32, 8, 1 << 20, 128, 7) == 7


def _topdelta_splits(fd, B, Hq, Hkv, L, d=128):
    """Chunks per sequence the top-delta planner picks, read back from its
    workspace size: the partials of B x Hq x S rows of d + 2 floats, plus 256
    bytes of alignment slack."""
    ws = fd.fd_topdelta_workspace_size(B, Hq, Hkv, L, d)
    per_chunk = B * Hq * (d + 2) * 4
    assert ws > 256 and (ws - 256) % per_chunk == 0, ws
    return (ws - 256) // per_chunk


def test_topdelta_workspace_decodes_explicit_counts(fd):
    for S in (2, 9, 19, 38):
        assert fd.fd_topdelta_workspace_size(4, 32, 8, 131072, 128, S) == S * 4 * 32 * 130 * 4 + 256


@pytest.mark.parametrize("B,Hq,Hkv,L", [(4, 32, 8, 131072), (1, 32, 8, 65536)])
def test_topdelta_plan_one_wave(fd, B, Hq, Hkv, L):
    slots = TOPDELTA_CTAS_PER_SM * _sms()
    S = _topdelta_splits(fd, B, Hq, Hkv, L)
    ctas = B * Hkv * S
    assert ctas <= slots, (S, ctas, slots)
    assert ctas + B * Hkv > slots, (S, ctas, slots)
