"""ctypes binding of libmoe_tsg.so: the C ABI of include/moe_tsg.h, same names.

Argument marshalling only. Every step of the path runs in the library's CUDA
kernels; there is no Python or CPU fallback. Importing this module fails loudly
when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_tsg.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "moe_tsg.h")

MOE_MAX_RANKS = 8


class MoeError(RuntimeError):
    pass


class moe_cfg(ctypes.Structure):
    _fields_ = [
        ("W", ctypes.c_int),
        ("L", ctypes.c_int),
        ("topk", ctypes.c_int),
        ("T", ctypes.c_int),
        ("d_model", ctypes.c_int),
        ("d_ff", ctypes.c_int),
        ("tb_M", ctypes.c_int),
        ("mgb", ctypes.c_int),
        ("consumer_ctas", ctypes.c_int),
        ("timeout_ns", ctypes.c_longlong),
        ("producer_pairs", ctypes.c_int),
    ]


def _parse_enums():
    """Enum constants of the header (MOE_OK, MOE_PLAN_*, MOE_RANK_*, ...)."""
    text = open(HEADER).read()
    out = {}
    for body in re.findall(r"enum\s+\w+\s*\{(.*?)\};", text, re.S):
        body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
        val = -1
        for item in body.split(","):
            item = item.strip()
            if not item:
                continue
            if "=" in item:
                name, v = (x.strip() for x in item.split("="))
                val = int(v)
            else:
                name, val = item, val + 1
            out[name] = val
    return out


ENUMS = _parse_enums()
globals().update(ENUMS)
# Integer #defines of the header (MOE_MAX_RANKS, MOE_CONSUMER_FUSED, ...).
DEFINES = {n: int(v) for n, v in re.findall(r"#define\s+(MOE_\w+)\s+\(?(-?\d+)\)?", open(HEADER).read())}
globals().update(DEFINES)


def load():
    if not os.path.exists(LIB_PATH):
        raise MoeError(
            f"{LIB_PATH} is missing: the CUDA library is not built "
            "(run tile_signaled_grouped_gb300.build.build() or __graft_entry__.build())")
    lib = ctypes.CDLL(LIB_PATH)
    vp, ip, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "moe_workspace_size": (ip, [P(moe_cfg), P(sz), P(sz), P(ip)]),
        "moe_plan_create": (ip, [P(moe_cfg), vp, sz, P(vp), sz, P(vp)]),
        "moe_plan_destroy": (None, [vp]),
        "moe_route": (ip, [vp, vp, vp, vp, vp, vp]),
        "moe_gate": (ip, [vp, P(vp), vp, vp, vp, vp, vp, ip, vp]),
        "moe_plan_build": (ip, [vp, vp, P(vp), vp]),
        "moe_expert_combine": (ip, [vp, P(vp), P(vp), P(vp), P(vp), vp, vp]),
        "moe_scale": (ip, [vp, vp, P(vp), P(vp), vp]),
        "moe_scale_gated": (ip, [vp, vp, P(vp), P(vp), vp]),
        "moe_producer_spans": (ip, [vp, P(ctypes.c_ulonglong), P(ctypes.c_ulonglong), ip, P(ip)]),
        "moe_combine_overlap": (ip, [vp, P(ctypes.c_double), P(ctypes.c_double),
                                     P(ctypes.c_double)]),
        "moe_status": (ip, [vp, vp, P(ip), P(ip)]),
        "moe_status_clear": (ip, [vp, vp]),
        "moe_field": (ip, [P(moe_cfg), ip, P(sz), P(sz)]),
        "moe_set_timing": (ip, [vp, ip]),
        "moe_timings": (ip, [vp, P(ctypes.c_float), ip]),
        "moe_plan_build_noalloc": (ip, [P(moe_cfg), vp, vp, sz, vp]),
        "moe_launch_info": (ip, [vp, P(ip), P(ip), P(ip), P(ip)]),
        "moe_set_schedule": (ip, [vp, ip, ip]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = load()
    return _lib


def check(rc: int, what: str):
    if rc != 0:
        names = {v: k for k, v in ENUMS.items() if k.startswith("MOE_ERR") or k == "MOE_OK"}
        raise MoeError(f"{what} failed: {names.get(rc, rc)}")


def ptr_array(ptrs):
    arr = (ctypes.c_void_p * MOE_MAX_RANKS)()
    for i, p in enumerate(ptrs):
        arr[i] = p
    return arr


# Thin wrappers with the C names --------------------------------------------

def moe_workspace_size(cfg: moe_cfg):
    pb, rb, rr = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_int()
    check(lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(pb), ctypes.byref(rb),
                                   ctypes.byref(rr)), "moe_workspace_size")
    return pb.value, rb.value, rr.value


def moe_field(cfg: moe_cfg, field: int):
    off, cnt = ctypes.c_size_t(), ctypes.c_size_t()
    check(lib().moe_field(ctypes.byref(cfg), field, ctypes.byref(off), ctypes.byref(cnt)),
          "moe_field")
    return off.value, cnt.value


def moe_plan_create(cfg: moe_cfg, plan_ws: int, plan_bytes: int, rank_ws, rank_bytes: int):
    out = ctypes.c_void_p()
    check(lib().moe_plan_create(ctypes.byref(cfg), plan_ws, plan_bytes, ptr_array(rank_ws),
                                rank_bytes, ctypes.byref(out)), "moe_plan_create")
    return out.value


def moe_plan_destroy(plan: int):
    lib().moe_plan_destroy(plan)


def moe_route(plan, logits, forced_ids, topk_ids, topk_w, stream):
    check(lib().moe_route(plan, logits, forced_ids, topk_ids, topk_w, stream), "moe_route")


def moe_gate(plan, x, w_router, forced_ids, topk_ids, topk_w, logits, splits, stream):
    check(lib().moe_gate(plan, ptr_array(x), w_router, forced_ids, topk_ids, topk_w, logits,
                         splits, stream), "moe_gate")


def moe_plan_build(plan, topk_ids, x, stream):
    check(lib().moe_plan_build(plan, topk_ids, ptr_array(x), stream), "moe_plan_build")


def moe_expert_combine(plan, w_gate, w_up, w_down, recv, producer, consumer):
    check(lib().moe_expert_combine(plan, ptr_array(w_gate), ptr_array(w_up), ptr_array(w_down),
                                   ptr_array(recv), producer, consumer), "moe_expert_combine")


def moe_scale(plan, topk_w, recv, out, stream):
    check(lib().moe_scale(plan, topk_w, ptr_array(recv), ptr_array(out), stream), "moe_scale")


def moe_scale_gated(plan, topk_w, recv, out, stream):
    check(lib().moe_scale_gated(plan, topk_w, ptr_array(recv), ptr_array(out), stream),
          "moe_scale_gated")


def moe_producer_spans(plan, max_records=1024):
    """[(start_ns, end_ns)] of the recorded producer launches, oldest first."""
    s = (ctypes.c_ulonglong * max_records)()
    e = (ctypes.c_ulonglong * max_records)()
    n = ctypes.c_int()
    check(lib().moe_producer_spans(plan, s, e, max_records, ctypes.byref(n)), "moe_producer_spans")
    return [(s[i], e[i]) for i in range(n.value)]


def moe_combine_overlap(plan):
    """(landed_frac, tail_us, copy_bytes) of the last recorded combine."""
    v = [ctypes.c_double() for _ in range(3)]
    check(lib().moe_combine_overlap(plan, *[ctypes.byref(x) for x in v]), "moe_combine_overlap")
    return tuple(x.value for x in v)


def moe_status(plan, stream):
    code, detail = ctypes.c_int(), ctypes.c_int()
    check(lib().moe_status(plan, stream, ctypes.byref(code), ctypes.byref(detail)), "moe_status")
    return code.value, detail.value


def moe_status_clear(plan, stream):
    check(lib().moe_status_clear(plan, stream), "moe_status_clear")


def moe_set_timing(plan, mode):
    """mode: 0/False off, 1/True CUDA events and device-clock records, 2 device clock only."""
    check(lib().moe_set_timing(plan, int(mode)), "moe_set_timing")


def moe_timings(plan, n: int = 6):
    buf = (ctypes.c_float * n)()
    check(lib().moe_timings(plan, buf, n), "moe_timings")
    return list(buf)


def moe_plan_build_noalloc(cfg: moe_cfg, topk_ids, plan_out, plan_out_bytes, stream):
    check(lib().moe_plan_build_noalloc(ctypes.byref(cfg), topk_ids, plan_out, plan_out_bytes,
                                       stream), "moe_plan_build_noalloc")


def moe_launch_info(plan):
    """(producer_ctas, consumer_ctas, num_sms, pair_clusters) of the overlapped schedule."""
    v = [ctypes.c_int() for _ in range(4)]
    check(lib().moe_launch_info(plan, *[ctypes.byref(x) for x in v]), "moe_launch_info")
    return tuple(x.value for x in v)


def moe_set_schedule(plan, consumer_ctas: int, mgb: int):
    check(lib().moe_set_schedule(plan, consumer_ctas, mgb), "moe_set_schedule")
