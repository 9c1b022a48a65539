"""The C ABI on a machine without a GPU: the library builds, loads and exports
every function include/moe_tsg.h declares; the host-side arithmetic and
argument checks behave as documented. No kernel is launched."""
import ctypes
import os
import re

import pytest

from tile_signaled_grouped_gb300 import build as B
from tile_signaled_grouped_gb300 import capi

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe_tsg.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return capi.load()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|void)\s+\**\s*(moe_\w+)\s*\(", text, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in ["moe_plan_build", "moe_expert_combine", "moe_scale", "moe_route"]:
        assert n in names
    raw = ctypes.CDLL(B.LIB)
    for n in names:
        assert hasattr(raw, n), f"{n} declared but not exported"


def _cfg(**kw):
    base = dict(W=4, L=2, topk=2, T=4096, d_model=2048, d_ff=8192, tb_M=128, mgb=1,
                consumer_ctas=8, timeout_ns=0, producer_pairs=0)
    base.update(kw)
    return capi.moe_cfg(*[base[f] for f, _ in capi.moe_cfg._fields_])


def test_workspace_sizes_follow_the_worst_case(lib):
    c = _cfg()
    plan_bytes, rank_bytes, recv_rows = capi.moe_workspace_size(c)
    assert recv_rows == 4096 * 2  # every token's k outputs could come back
    # worst-case rows of one owner: W*T*min(k,L) + L*W*(tb-1), rounded to tb
    rm = 4 * 4096 * 2 + 2 * 4 * 127
    rm = -(-rm // 128) * 128
    assert rank_bytes == rm * 2048 * 2 * 2 + rm * 8192 * 2
    off_x, n_x = capi.moe_field(c, capi.MOE_RANK_X)
    off_h, n_h = capi.moe_field(c, capi.MOE_RANK_H)
    off_y, n_y = capi.moe_field(c, capi.MOE_RANK_Y)
    assert (off_x, n_x) == (0, rm * 2048) and off_h == rm * 2048 * 2
    assert off_y == off_h + rm * 8192 * 2 and n_y == rm * 2048
    # plan fields lie inside the plan workspace and do not overlap
    spans = []
    for name, v in capi.ENUMS.items():
        if name.startswith("MOE_PLAN_") and name != "MOE_PLAN_NFIELDS":
            off, cnt = capi.moe_field(c, v)
            assert off + 4 * cnt <= plan_bytes, name
            spans.append((off, off + 4 * cnt, name))
    spans.sort()
    for (a0, a1, na), (b0, b1, nb) in zip(spans, spans[1:]):
        assert a1 <= b0, (na, nb)


@pytest.mark.parametrize("bad", [
    dict(W=0), dict(W=9), dict(L=0), dict(topk=0), dict(topk=9, W=1, L=8), dict(T=0),
    dict(d_model=100), dict(d_ff=64), dict(tb_M=96), dict(mgb=0), dict(consumer_ctas=-1),
    dict(producer_pairs=2), dict(producer_pairs=-1),
    dict(consumer_ctas=-1, producer_pairs=0), dict(consumer_ctas=-2, producer_pairs=1),
])
def test_invalid_configurations_are_rejected(lib, bad):
    with pytest.raises(capi.MoeError, match="MOE_ERR_ARG"):
        capi.moe_workspace_size(_cfg(**bad))


def test_token_rows_must_fit_one_copy_chunk(lib):
    # The combine copy moves whole rows through 20 KB shared-memory slots.
    assert capi.moe_workspace_size(_cfg(d_model=10240))[0] > 0
    with pytest.raises(capi.MoeError, match="MOE_ERR_UNSUPPORTED"):
        capi.moe_workspace_size(_cfg(d_model=10240 + 128))


def test_cfg_struct_matches_the_header(lib):
    """The ctypes mirror of moe_cfg has the header's fields in the header's order."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct moe_cfg \{(.*?)\} moe_cfg;", text, re.S).group(1)
    names = re.findall(r"(\w+);", body)
    assert names == [f for f, _ in capi.moe_cfg._fields_]
    assert ctypes.sizeof(capi.moe_cfg) == 56


def test_host_errors_without_a_device(lib):
    c = _cfg(W=2, L=2, T=64, d_model=128, d_ff=128, tb_M=64)
    pb, rb, _ = capi.moe_workspace_size(c)
    # misaligned or missing workspaces are argument errors, checked before any CUDA call
    with pytest.raises(capi.MoeError, match="MOE_ERR_ARG"):
        capi.moe_plan_create(c, 0, pb, [1024, 2048], rb)
    with pytest.raises(capi.MoeError, match="MOE_ERR_ARG"):
        capi.moe_plan_create(c, 1024, pb, [1024 + 16, 4096], rb)
    with pytest.raises(capi.MoeError, match="MOE_ERR_WORKSPACE"):
        capi.moe_plan_create(c, 1024, pb - 1, [1024, 4096], rb)
    # well-formed arguments reach the runtime, which finds no sm_103 device here
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if not has_gpu:
        with pytest.raises(capi.MoeError, match="MOE_ERR_CUDA|MOE_ERR_UNSUPPORTED"):
            capi.moe_plan_create(c, 1024, pb, [1024, 4096], rb)
    # calls on a null plan are argument errors
    lib_ = capi.lib()
    assert lib_.moe_plan_build(None, None, None, None) == capi.MOE_ERR_ARG
    assert lib_.moe_scale(None, None, None, None, None) == capi.MOE_ERR_ARG
    assert lib_.moe_set_timing(None, 1) == capi.MOE_ERR_ARG


@pytest.mark.parametrize("shape", [
    dict(W=3, L=3, topk=2, T=77, d_model=256, d_ff=384, tb_M=64, mgb=3),
    dict(W=4, L=2, topk=3, T=130, d_model=128, d_ff=256, tb_M=128),
    dict(W=8, L=32, topk=8, T=256, d_model=7168, d_ff=2048, tb_M=64),
    dict(W=1, L=3, topk=2, T=50, d_model=128, d_ff=256, tb_M=128),
])
def test_plan_arrays_are_aligned(lib, shape):
    """Kernels read plan arrays with 16-byte vector loads: every array outside the
    packed per-combine region (ready flags, group signals) starts on 256 bytes."""
    c = _cfg(**shape)
    for name, v in capi.ENUMS.items():
        if name.startswith("MOE_PLAN_") and name not in ("MOE_PLAN_NFIELDS", "MOE_PLAN_FLAGS",
                                                         "MOE_PLAN_GROUP_SIG"):
            off, _ = capi.moe_field(c, v)
            assert off % 256 == 0, (name, off)


def test_fused_schedule_is_a_valid_configuration(lib):
    """consumer_ctas = MOE_CONSUMER_FUSED needs the pair producer; then it is accepted."""
    assert capi.MOE_CONSUMER_FUSED == -1
    pb, rb, _ = capi.moe_workspace_size(_cfg(consumer_ctas=capi.MOE_CONSUMER_FUSED,
                                             producer_pairs=1))
    assert pb > 0 and rb > 0


def test_plan_calls_reject_a_null_plan(lib):
    lib_ = capi.lib()
    assert lib_.moe_set_schedule(None, 0, 1) == capi.MOE_ERR_ARG
    assert lib_.moe_launch_info(None, None, None, None, None) == capi.MOE_ERR_ARG
    assert lib_.moe_status(None, None, None, None) == capi.MOE_ERR_ARG
    assert lib_.moe_gate(None, None, None, None, None, None, None, 0, None) == capi.MOE_ERR_ARG
