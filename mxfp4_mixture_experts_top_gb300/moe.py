"""Python binding of the C ABI in include/moe_mxfp4.h (ctypes).

Argument marshalling only: every step of the layer runs in the CUDA library
libmoe_mxfp4.so. PyTorch provides device memory and the current stream. There
is no fallback: if the library has not been built, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_mxfp4.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_MISALIGNED",
                4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_DEVICE", 7: "MOE_ERR_TIMEOUT"}

# Every symbol the header declares (checked by the CPU test suite).
EXPORTS = ["moe_abi_version", "moe_status_string", "moe_route", "moe_permute_rows_capacity", "moe_permute",
           "moe_mxfp4_packed_bytes", "moe_mxfp4_prepack", "moe_mxfp4_dequant_bf16", "moe_mxfp4_workspace_bytes",
           "moe_mxfp4_forward", "moe_mxfp4_forward_timed", "moe_mxfp4_workspace_layout", "moe_mxfp4_forward_plan", "moe_read_device_error", "moe_launch_count",
           "moe_selftest_bounded_wait",
           "moe_mxfp4_forward_noalloc", "moe_route_permute", "moe_permute_workspace_size", "moe_clear_cache",
           "moe_mxfp4_noalloc_read_device_error", "moe_ep_dispatch_pack", "moe_ep_combine"]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({_lib_status_string(status)})")


class LayerDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int),
                ("k", ctypes.c_int), ("block_m", ctypes.c_int), ("swiglu_limit", ctypes.c_float),
                ("out_dtype", ctypes.c_int), ("flags", ctypes.c_uint)]


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH):
    """Load libmoe_mxfp4.so; raises if it is missing (build it with __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        D = ctypes.POINTER(LayerDesc)
        sigs = {
            "moe_abi_version": ([], i32),
            "moe_status_string": ([i32], ctypes.c_char_p),
            "moe_route": ([P, i32, i32, i32, P, P, P, P], i32),
            "moe_permute_rows_capacity": ([i32, i32, i32, i32], i64),
            "moe_permute": ([P, i32, i32, i32, i32, P, P, P, P, P, P, P], i32),
            "moe_mxfp4_packed_bytes": ([D], sz),
            "moe_mxfp4_prepack": ([D, P, P, P, P, P, sz, P], i32),
            "moe_mxfp4_dequant_bf16": ([D, P, i32, i32, P, P], i32),
            "moe_mxfp4_workspace_bytes": ([D], sz),
            "moe_mxfp4_forward": ([D, P, P, P, P, P, P, P, P, sz, P], i32),
            "moe_mxfp4_forward_timed": ([D, P, P, P, P, P, P, P, P, sz, P, P], i32),
            "moe_mxfp4_workspace_layout": ([D, ctypes.POINTER(ctypes.c_size_t * 7)], i32),
            "moe_mxfp4_forward_plan": ([D, ctypes.POINTER(ctypes.c_int * 4)], i32),
            "moe_read_device_error": ([P, ctypes.POINTER(ctypes.c_int), P], i32),
            "moe_launch_count": ([], ctypes.c_uint64),
            "moe_selftest_bounded_wait": ([ctypes.c_uint64, ctypes.c_uint64, P, P, P], i32),
            "moe_mxfp4_forward_noalloc": ([D, P, P, P, P, P, P, P, P], i32),
            "moe_route_permute": ([P, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P], i32),
            "moe_permute_workspace_size": ([i32, i32, i32, i32], sz),
            "moe_clear_cache": ([], None),
            "moe_mxfp4_noalloc_read_device_error": ([ctypes.POINTER(ctypes.c_int), P], i32),
            "moe_ep_dispatch_pack": ([P, i32, i32, i32, i32, i32, P, P, P, P, P, P], i32),
            "moe_ep_combine": ([P, i32, i32, i32, i32, P, P, P, P, P, P, P, P], i32),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _lib_status_string(status: int) -> str:
    try:
        return load().moe_status_string(status).decode()
    except Exception:  # pragma: no cover - only while formatting an error
        return "?"


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
    return t


def abi_version() -> int:
    return load().moe_abi_version()


def launch_count() -> int:
    return int(load().moe_launch_count())


def rows_capacity(T: int, E: int, k: int, block_m: int) -> int:
    return int(load().moe_permute_rows_capacity(T, E, k, block_m))


def route(logits: torch.Tensor, k: int, bitmatrix: bool = True, out=None, stream=None):
    """moe_route. Returns (topk_ids int32 [T,k], topk_w fp32 [T,k], bitmatrix int32 [T, ceil(E/32)] or None)."""
    _cuda(logits, torch.float32, "logits")
    T, E = logits.shape
    if out is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
        w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
        bm = torch.empty((T, (E + 31) // 32), dtype=torch.int32, device=logits.device) if bitmatrix else None
    else:
        ids, w, bm = out
    _check(load().moe_route(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _ptr(bm), _stream(stream)), "moe_route")
    return ids, w, bm


def permute(topk_ids: torch.Tensor, E: int, block_m: int, out=None, error=None, stream=None):
    """moe_permute. Returns dict counts, offsets, padded_offsets, row_to_pair, pair_to_row (int32)."""
    _cuda(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    dev = topk_ids.device
    if out is None:
        cap = rows_capacity(T, E, k, block_m)
        out = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   padded_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   row_to_pair=torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
                   pair_to_row=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev))
    _check(load().moe_permute(_ptr(topk_ids), T, E, k, block_m, _ptr(out["counts"]), _ptr(out["offsets"]),
                              _ptr(out["padded_offsets"]), _ptr(out["row_to_pair"]), _ptr(out["pair_to_row"]),
                              _ptr(error), _stream(stream)), "moe_permute")
    return out


def route_permute(logits: torch.Tensor, k: int, block_m: int, out=None, perm_out=None, error=None, stream=None):
    """moe_route_permute (one launch for T <= 128). Returns (topk_ids, topk_w, bitmatrix, perm dict)."""
    _cuda(logits, torch.float32, "logits")
    T, E = logits.shape
    dev = logits.device
    if out is None:
        out = (torch.empty((T, k), dtype=torch.int32, device=dev), torch.empty((T, k), dtype=torch.float32, device=dev),
               torch.empty((T, (E + 31) // 32), dtype=torch.int32, device=dev))
    ids, w, bm = out
    if perm_out is None:
        cap = rows_capacity(T, E, k, block_m)
        perm_out = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
                        offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                        padded_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                        row_to_pair=torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
                        pair_to_row=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev))
    po = perm_out
    _check(load().moe_route_permute(_ptr(logits), T, E, k, block_m, _ptr(ids), _ptr(w), _ptr(bm), _ptr(po["counts"]),
                                    _ptr(po["offsets"]), _ptr(po["padded_offsets"]), _ptr(po["row_to_pair"]),
                                    _ptr(po["pair_to_row"]), _ptr(error), _stream(stream)), "moe_route_permute")
    return ids, w, bm, po


FLAG_FAST_COMBINE = 1   # MOE_FLAG_FAST_COMBINE
OUT_F32, OUT_BF16 = 0, 1  # moe_out_dtype_t


def make_desc(T, H, I, E, k, block_m=16, swiglu_limit=0.0, flags=0, out_dtype=OUT_F32) -> LayerDesc:
    return LayerDesc(T, H, I, E, k, block_m, float(swiglu_limit), int(out_dtype), int(flags))


def packed_bytes(desc: LayerDesc) -> int:
    return int(load().moe_mxfp4_packed_bytes(ctypes.byref(desc)))


def workspace_bytes(desc: LayerDesc) -> int:
    return int(load().moe_mxfp4_workspace_bytes(ctypes.byref(desc)))


def workspace_layout(desc: LayerDesc):
    arr = (ctypes.c_size_t * 7)()
    _check(load().moe_mxfp4_workspace_layout(ctypes.byref(desc), ctypes.byref(arr)), "moe_mxfp4_workspace_layout")
    return dict(error=arr[0], xq=arr[1], xs=arr[2], hq=arr[3], hs=arr[4], staging=arr[5], total=arr[6])


REGIMES = ("tiny", "small", "mid", "large", "huge")


def forward_plan(desc: LayerDesc):
    """moe_mxfp4_forward_plan: the tile regime, whether W13 and W2 run as one launch, whether the
    atomic combine is taken, and the number of kernels moe_mxfp4_forward launches."""
    arr = (ctypes.c_int * 4)()
    _check(load().moe_mxfp4_forward_plan(ctypes.byref(desc), ctypes.byref(arr)), "moe_mxfp4_forward_plan")
    return dict(regime=REGIMES[arr[0]], fused_gemms=bool(arr[1]), fast_combine=bool(arr[2]), launches=arr[3])


def prepack(desc: LayerDesc, w13_q, w13_s, w2_q, w2_s, stream=None) -> torch.Tensor:
    """moe_mxfp4_prepack into a new uint8 device buffer."""
    for t, n in ((w13_q, "w13_q"), (w13_s, "w13_s"), (w2_q, "w2_q"), (w2_s, "w2_s")):
        _cuda(t, torch.uint8, n)
    nbytes = packed_bytes(desc)
    packed = torch.empty(nbytes, dtype=torch.uint8, device=w13_q.device)
    _check(load().moe_mxfp4_prepack(ctypes.byref(desc), _ptr(w13_q), _ptr(w13_s), _ptr(w2_q), _ptr(w2_s),
                                    _ptr(packed), nbytes, _stream(stream)), "moe_mxfp4_prepack")
    return packed


def dequant_bf16(desc: LayerDesc, packed: torch.Tensor, which: int, expert: int, stream=None) -> torch.Tensor:
    """moe_mxfp4_dequant_bf16: one expert's W13 ([2I, H]) or W2 ([H, I]) as bf16."""
    shape = (2 * desc.I, desc.H) if which == 0 else (desc.H, desc.I)
    out = torch.empty(shape, dtype=torch.bfloat16, device=packed.device)
    _check(load().moe_mxfp4_dequant_bf16(ctypes.byref(desc), _ptr(packed), which, expert, _ptr(out),
                                         _stream(stream)), "moe_mxfp4_dequant_bf16")
    return out


def forward(desc: LayerDesc, x: torch.Tensor, packed: torch.Tensor, topk_w: torch.Tensor, perm: dict,
            workspace: torch.Tensor, y: torch.Tensor = None, stream=None) -> torch.Tensor:
    """moe_mxfp4_forward: y fp32 [T, H]."""
    _cuda(x, torch.bfloat16, "x")
    ydt = torch.bfloat16 if desc.out_dtype == OUT_BF16 else torch.float32
    if y is None:
        y = torch.empty((desc.T, desc.H), dtype=ydt, device=x.device)
    _cuda(y, ydt, "y")
    _check(load().moe_mxfp4_forward(ctypes.byref(desc), _ptr(x), _ptr(packed), _ptr(topk_w), _ptr(perm["offsets"]),
                                    _ptr(perm["padded_offsets"]), _ptr(perm["row_to_pair"]), _ptr(y),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream)), "moe_mxfp4_forward")
    return y


NOALLOC_SCRATCH_BYTES = 32 << 20   # MOE_NOALLOC_SCRATCH_BYTES


def forward_noalloc(desc: LayerDesc, x: torch.Tensor, packed: torch.Tensor, topk_w: torch.Tensor, perm: dict,
                    y: torch.Tensor = None, stream=None) -> torch.Tensor:
    """moe_mxfp4_forward_noalloc: the forward with the library's static scratch array as its
    workspace, for callers that cannot allocate device memory (y must be passed in then)."""
    _cuda(x, torch.bfloat16, "x")
    ydt = torch.bfloat16 if desc.out_dtype == OUT_BF16 else torch.float32
    if y is None:
        y = torch.empty((desc.T, desc.H), dtype=ydt, device=x.device)
    _cuda(y, ydt, "y")
    _check(load().moe_mxfp4_forward_noalloc(ctypes.byref(desc), _ptr(x), _ptr(packed), _ptr(topk_w),
                                            _ptr(perm["offsets"]), _ptr(perm["padded_offsets"]),
                                            _ptr(perm["row_to_pair"]), _ptr(y), _stream(stream)),
           "moe_mxfp4_forward_noalloc")
    return y


def forward_timed(desc: LayerDesc, x: torch.Tensor, packed: torch.Tensor, topk_w: torch.Tensor, perm: dict,
                  workspace: torch.Tensor, y: torch.Tensor, events, stream=None) -> torch.Tensor:
    """moe_mxfp4_forward_timed: records 5 torch.cuda.Event objects between the forward's kernels."""
    arr = (ctypes.c_void_p * 5)(*[ctypes.c_void_p(e.cuda_event) if e is not None else None for e in events])
    _check(load().moe_mxfp4_forward_timed(ctypes.byref(desc), _ptr(x), _ptr(packed), _ptr(topk_w),
                                          _ptr(perm["offsets"]), _ptr(perm["padded_offsets"]),
                                          _ptr(perm["row_to_pair"]), _ptr(y), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), arr, _stream(stream)),
           "moe_mxfp4_forward_timed")
    return y


def selftest_bounded_wait(limit_ns: int, abort_after_ns: int, error: torch.Tensor, elapsed: torch.Tensor,
                          stream=None) -> None:
    """moe_selftest_bounded_wait: a pipeline wait that nothing completes gives up (after limit_ns, or when
    another warp sets the abort flag after abort_after_ns) and records MOE_ERR_TIMEOUT in `error`."""
    _cuda(error, torch.int32, "error")
    _cuda(elapsed, torch.int64, "elapsed")
    _check(load().moe_selftest_bounded_wait(limit_ns, abort_after_ns, _ptr(error), _ptr(elapsed), _stream(stream)),
           "moe_selftest_bounded_wait")


def ep_dispatch_pack(x: torch.Tensor, perm: dict, k: int, experts_per_rank: int, send_x=None, send_ids=None,
                     stream=None):
    """moe_ep_dispatch_pack: the activation rows of the T*k pairs in (expert, token) order, and their
    experts as ids local to the owning rank. Returns (send_x bf16 [T*k, H], send_ids int32 [T*k])."""
    _cuda(x, torch.bfloat16, "x")
    T, H = x.shape
    E = perm["counts"].numel()
    if send_x is None:
        send_x = torch.empty((T * k, H), dtype=torch.bfloat16, device=x.device)
    if send_ids is None:
        send_ids = torch.empty(max(T * k, 1), dtype=torch.int32, device=x.device)
    _check(load().moe_ep_dispatch_pack(_ptr(x), T, H, E, k, experts_per_rank, _ptr(perm["offsets"]),
                                       _ptr(perm["padded_offsets"]), _ptr(perm["row_to_pair"]), _ptr(send_x),
                                       _ptr(send_ids), _stream(stream)), "moe_ep_dispatch_pack")
    return send_x, send_ids


def ep_combine(returned: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor, perm: dict, y=None, error=None,
               stream=None) -> torch.Tensor:
    """moe_ep_combine: y[t] = sum_j w[t, j] * returned[row of pair (t, j) in send order], slots ascending."""
    _cuda(returned, torch.float32, "returned")
    T, k = topk_ids.shape
    H = returned.shape[1]
    E = perm["counts"].numel()
    if y is None:
        y = torch.empty((T, H), dtype=torch.float32, device=returned.device)
    _check(load().moe_ep_combine(_ptr(returned), T, H, E, k, _ptr(topk_ids), _ptr(topk_w), _ptr(perm["offsets"]),
                                 _ptr(perm["padded_offsets"]), _ptr(perm["pair_to_row"]), _ptr(y), _ptr(error),
                                 _stream(stream)), "moe_ep_combine")
    return y


def noalloc_read_device_error(stream=None) -> int:
    """moe_mxfp4_noalloc_read_device_error: read and clear the error word of forward_noalloc."""
    code = ctypes.c_int(0)
    _check(load().moe_mxfp4_noalloc_read_device_error(ctypes.byref(code), _stream(stream)),
           "moe_mxfp4_noalloc_read_device_error")
    return code.value


def clear_cache() -> None:
    """moe_clear_cache: drop the library's host-side cache of TMA tensor maps."""
    load().moe_clear_cache()


def permute_workspace_size(T: int, E: int, k: int, block_m: int) -> int:
    return int(load().moe_permute_workspace_size(T, E, k, block_m))


def read_device_error(word: torch.Tensor, stream=None) -> int:
    """moe_read_device_error on a device int32 word (permute error word or workspace start)."""
    code = ctypes.c_int(0)
    _check(load().moe_read_device_error(_ptr(word), ctypes.byref(code), _stream(stream)), "moe_read_device_error")
    return code.value


@dataclass
class MoELayer:
    """One MXFP4 MoE layer on the current CUDA device: prepacked weights plus
    persistent buffers, so a call is route+permute (one launch for small
    batches) -> forward with no allocation (CUDA-graph capturable)."""

    desc: LayerDesc
    packed: torch.Tensor
    workspace: torch.Tensor
    bufs: dict

    @classmethod
    def create(cls, T, H, I, E, k, w13_q, w13_s, w2_q, w2_s, block_m=16, swiglu_limit=0.0, device="cuda",
               flags=0, out_dtype=OUT_F32):
        desc = make_desc(T, H, I, E, k, block_m, swiglu_limit, flags, out_dtype)
        packed = prepack(desc, w13_q, w13_s, w2_q, w2_s)
        ws = torch.empty(max(workspace_bytes(desc), 1024), dtype=torch.uint8, device=device)
        cap = rows_capacity(T, E, k, block_m)
        dev = torch.device(device)
        bufs = dict(ids=torch.empty((T, k), dtype=torch.int32, device=dev),
                    w=torch.empty((T, k), dtype=torch.float32, device=dev),
                    bm=torch.empty((T, (E + 31) // 32), dtype=torch.int32, device=dev),
                    perm=dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
                              offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                              padded_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                              row_to_pair=torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
                              pair_to_row=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)),
                    perm_err=torch.zeros(4, dtype=torch.int32, device=dev),
                    y=torch.empty((T, H), dtype=torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32,
                                  device=dev))
        return cls(desc, packed, ws, bufs)

    def __call__(self, x: torch.Tensor, logits: torch.Tensor, stream=None) -> torch.Tensor:
        b = self.bufs
        route_permute(logits, self.desc.k, self.desc.block_m, out=(b["ids"], b["w"], b["bm"]), perm_out=b["perm"],
                      error=b["perm_err"], stream=stream)
        return forward(self.desc, x, self.packed, b["w"], b["perm"], self.workspace, y=b["y"], stream=stream)

    def capture_graph(self, x: torch.Tensor, logits: torch.Tensor):
        """Capture route -> permute -> forward on x/logits (fixed addresses) into
        one CUDA graph; returns (graph, y). Replaying the graph re-runs the whole
        layer on whatever x and logits then hold, with one launch."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self(x, logits)                       # warm-up outside capture (sets kernel attributes)
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            y = self(x, logits)
        return graph, y

    def forward_error(self) -> int:
        return read_device_error(self.workspace[:4].view(torch.int32))
