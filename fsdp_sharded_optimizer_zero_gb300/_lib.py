"""ctypes binding of libzero_gb300.so: argument marshalling only.

Each function below has the name of the C entry point it calls. Tensors are torch CUDA
tensors (PyTorch supplies device memory and streams); the binding checks dtype, device and
contiguity, passes raw pointers and the current stream, and raises ZeroError on a
non-zero status. Every arithmetic step runs in the library's CUDA kernels; there is no
Python or CPU fallback: if the shared library is missing the import fails.
"""
from __future__ import annotations

import ctypes as C
import os
from pathlib import Path

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libzero_gb300.so"

ZERO_OK = 0
ZERO_ERR_INVALID_ARG = -1
ZERO_ERR_OOM = -2
ZERO_ERR_CUDA = -3
ZERO_ERR_UNSUPPORTED = -4
ZERO_ERR_DEVICE = -5
ZERO_RANK_VIEW = -1
ZERO_ALL_RANKS = -2
ZERO_MAX_RANKS = 64
STAGE_IDS = {"ddp": 0, "zero1": 1, "zero2": 2, "zero3": 3, "megatron": 4}

# every symbol declared in include/zero.h
EXPORTS = (
    "zero_plan", "zero_plan_query", "zero_bucket_range", "zero_plan_destroy", "zero_plan_check_memory",
    "zero_reduce_scatter", "zero_adam_step", "zero_fused_step", "zero_fused_step_host", "zero_fused_step_fp32_grads",
    "zero_fused_step_buckets", "zero_allgather_params", "ddp_allreduce",
    "fsdp_gather_rows", "fsdp_unit_forward", "fsdp_transpose_cat", "fsdp_unit_backward_workspace", "fsdp_unit_backward", "fsdp_mlp_forward",
    "fsdp_zero3_step_workspace", "fsdp_zero3_step", "fsdp_zero3_mlp_step_workspace", "fsdp_zero3_mlp_step",
    "fsdp_unit_forward_static_scratch",
    "zero_last_error", "zero_device_status", "zero_selftest_bounded_wait", "zero_set_fused_kernel", "zero_set_gemm_kernel", "zero_version",
)


class ZeroError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class zero_layout(C.Structure):
    _fields_ = [
        ("psi", C.c_uint64), ("psi_padded", C.c_uint64), ("shard_elems", C.c_uint64),
        ("bucket_bytes", C.c_uint64), ("bucket_elems", C.c_uint64), ("n_buckets", C.c_uint64),
        ("n_ranks", C.c_int32), ("stage", C.c_int32),
        ("state_param_bytes", C.c_uint64), ("state_grad_bytes", C.c_uint64),
        ("state_master_bytes", C.c_uint64), ("state_m_bytes", C.c_uint64), ("state_v_bytes", C.c_uint64),
        ("state_total_bytes", C.c_uint64),
        ("comm_reduce_scatter", C.c_uint64), ("comm_all_gather_fwd", C.c_uint64),
        ("comm_all_gather_bwd", C.c_uint64), ("comm_total", C.c_uint64),
        ("ring_sent_elems", C.c_uint64), ("fused_step_bytes", C.c_uint64),
    ]


class fsdp_unit_state(C.Structure):
    _fields_ = [("rows_out", C.c_int64), ("k_in", C.c_int64), ("plan", C.c_void_p), ("w", C.c_void_p),
                ("master", C.c_void_p), ("m", C.c_void_p), ("v", C.c_void_p), ("x", C.c_void_p), ("dy", C.c_void_p),
                ("dw", C.c_void_p)]


class fsdp_weight_state(C.Structure):
    _fields_ = [("plan", C.c_void_p), ("w", C.c_void_p), ("master", C.c_void_p), ("m", C.c_void_p),
                ("v", C.c_void_p)]


class fsdp_mlp_unit_state(C.Structure):
    _fields_ = [("d_model", C.c_int64), ("d_ff", C.c_int64), ("gate", fsdp_weight_state), ("up", fsdp_weight_state),
                ("down", fsdp_weight_state), ("x", C.c_void_p), ("gu", C.c_void_p), ("h", C.c_void_p),
                ("dy", C.c_void_p), ("dh", C.c_void_p), ("dgu", C.c_void_p), ("dw_gu", C.c_void_p),
                ("dw_down", C.c_void_p)]


FSDP_GATHER_MATERIALIZE = 1
FSDP_BACKWARD_PREFETCH = 2
FSDP_OVERLAP_OPTIMIZER = 4
FSDP_SEPARATE_OPTIMIZER = 8


class zero_adam(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
                ("weight_decay", C.c_float)]


def _load():
    if not LIB_PATH.exists():
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(nvcc, sm_103a). There is no fallback path.")
    lib = C.CDLL(str(LIB_PATH))
    P, I, U64, I64, VP = C.c_void_p, C.c_int, C.c_uint64, C.c_int64, C.c_void_p
    PP = C.POINTER(C.c_void_p)
    sig = {
        "zero_plan": (I, [U64, I, I, U64, C.POINTER(C.c_void_p)]),
        "zero_plan_query": (I, [P, C.POINTER(zero_layout)]),
        "zero_bucket_range": (I, [P, I, U64, C.POINTER(U64), C.POINTER(U64)]),
        "zero_plan_destroy": (I, [P]),
        "zero_plan_check_memory": (I, [P, I, U64, C.POINTER(U64), C.POINTER(U64)]),
        "zero_reduce_scatter": (I, [P, I, PP, VP, VP]),
        "zero_adam_step": (I, [P, I, VP, VP, VP, VP, VP, C.POINTER(zero_adam), I64, VP]),
        "zero_fused_step": (I, [P, I, PP, VP, VP, VP, VP, C.POINTER(zero_adam), I64, VP]),
        "zero_fused_step_fp32_grads": (I, [P, I, PP, VP, VP, VP, VP, C.POINTER(zero_adam), I64, VP]),
        "zero_fused_step_host": (I, [P, I, PP, VP, VP, VP, VP, C.POINTER(zero_adam), I64, VP]),
        "zero_fused_step_buckets": (I, [P, I, U64, U64, PP, VP, VP, VP, VP, C.POINTER(zero_adam), I64, VP]),
        "zero_allgather_params": (I, [P, PP, VP, VP]),
        "ddp_allreduce": (I, [P, PP, VP, VP]),
        "fsdp_gather_rows": (I, [I, PP, I64, I64, VP, VP]),
        "fsdp_unit_forward": (I, [I, PP, I64, I64, VP, I64, VP, VP, VP, VP]),
        "fsdp_unit_forward_static_scratch": (I, [I, PP, I64, I64, VP, I64, VP, VP, VP]),
        "fsdp_transpose_cat": (I, [I, PP, I64, I64, VP, VP]),
        "fsdp_unit_backward_workspace": (I, [I, I64, I64, I64, C.POINTER(U64)]),
        "fsdp_unit_backward": (I, [I, PP, I64, I64, PP, PP, I64, PP, VP, VP, U64, VP]),
        "fsdp_mlp_forward": (I, [I, PP, PP, PP, I64, I64, VP, I64, VP, VP, VP, VP, VP]),
        "zero_last_error": (C.c_char_p, []),
        "zero_device_status": (I, [VP]),
        "zero_selftest_bounded_wait": (I, [C.c_uint32, VP]),
        "zero_set_fused_kernel": (I, [I]),
        "fsdp_zero3_step_workspace": (I, [I, I, C.POINTER(fsdp_unit_state), I64, I, C.POINTER(U64)]),
        "fsdp_zero3_step": (I, [I, I, C.POINTER(fsdp_unit_state), I64, VP, VP, C.POINTER(zero_adam), I64, I, VP, U64,
                                VP, VP]),
        "fsdp_zero3_mlp_step_workspace": (I, [I, I, C.POINTER(fsdp_mlp_unit_state), I64, C.POINTER(U64)]),
        "fsdp_zero3_mlp_step": (I, [I, I, C.POINTER(fsdp_mlp_unit_state), I64, VP, VP, C.POINTER(zero_adam), I64, I,
                                    VP, U64, VP]),
        "zero_set_gemm_kernel": (I, [I]),
        "zero_version": (I, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib


_lib = _load()


def _check(rc: int):
    if rc != ZERO_OK:
        raise ZeroError(rc, _lib.zero_last_error().decode(errors="replace"))


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.device.index is not None and t.device.index != torch.cuda.current_device():
        # the kernels run on the current device: another device's pointer would fault there
        raise ValueError(f"{name} is on {t.device}, the current device is cuda:{torch.cuda.current_device()}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _ptr_array(ts, dtype, name):
    arr = (C.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = _dev(t, dtype, f"{name}[{i}]")
    return arr


def _adam(hp) -> zero_adam:
    if isinstance(hp, zero_adam):
        return hp
    d = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    if hp is not None:
        d.update({k: getattr(hp, k) for k in d if hasattr(hp, k)} if not isinstance(hp, dict) else hp)
    return zero_adam(**d)


class Plan:
    """Owns a zero_plan_t handle."""

    def __init__(self, handle: int):
        self.handle = C.c_void_p(handle)
        self.layout = zero_plan_query(self)

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h and _lib is not None:
            _lib.zero_plan_destroy(h)

    def __getattr__(self, k):
        lay = self.__dict__.get("layout")
        if lay is not None and k in lay:
            return lay[k]
        raise AttributeError(k)


# ---------------------------------------------------------------------------------------
# buffer sizes: the C ABI takes raw pointers, so the binding checks every tensor's length
# against the plan (or the FSDP shapes) before anything is launched; a short buffer would
# otherwise be written past its end on the device
# ---------------------------------------------------------------------------------------

def _need(t, n: int, name: str):
    if t is not None and t.numel() < n:
        raise ValueError(f"{name} holds {t.numel()} elements; this call needs at least {n}")


def _step_sizes(plan: "Plan", rank: int):
    """Elements of (each rank's gradient, g / master / m / v, param_out) for `rank`, from
    the header's pointer conventions; zeros for a rank the library itself will reject."""
    P, S = plan.psi_padded, plan.shard_elems
    if rank == ZERO_ALL_RANKS:
        return P, P, P
    if rank == ZERO_RANK_VIEW:
        return S, S, S
    if 0 <= rank < plan.n_ranks:
        return P, S, (S if plan.stage == STAGE_IDS["zero3"] else P)
    return 0, 0, 0


def _check_step(plan: "Plan", rank: int, grads=None, state=(), param_out=None):
    ng, ns, npar = _step_sizes(plan, rank)
    if grads is not None:
        if len(grads) != plan.n_ranks:
            raise ValueError(f"grads holds {len(grads)} rank buffers; the plan has {plan.n_ranks} ranks")
        for i, g in enumerate(grads):
            _need(g, ng, f"grads[{i}]")
    for name, t in state:
        _need(t, ns, name)
    _need(param_out, npar, "param_out")


def _shards_shape(shards, name: str):
    """(rows of one shard, columns): every shard the same 2-D shape."""
    shapes = {tuple(s.shape) for s in shards}
    if len(shapes) != 1 or len(next(iter(shapes))) != 2:
        raise ValueError(f"{name} must be 2-D tensors of one shape (got {sorted(shapes)})")
    return next(iter(shapes))


# ---------------------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------------------

def zero_plan(psi: int, n_ranks: int, stage, bucket_bytes: int) -> Plan:
    stage = STAGE_IDS.get(stage, stage)
    h = C.c_void_p()
    _check(_lib.zero_plan(psi, n_ranks, stage, bucket_bytes, C.byref(h)))
    return Plan(h.value)


def zero_plan_query(plan: Plan) -> dict:
    lay = zero_layout()
    _check(_lib.zero_plan_query(plan.handle, C.byref(lay)))
    return {name: getattr(lay, name) for name, _ in zero_layout._fields_}


def zero_plan_check_memory(plan: Plan, rank: int, budget_bytes: int = 0):
    """(need, budget) in bytes for one step call of the plan in rank mode `rank`; raises
    ZeroError with code ZERO_ERR_OOM when need > budget (budget 0 = the device's free
    memory)."""
    need, budget = C.c_uint64(), C.c_uint64()
    _check(_lib.zero_plan_check_memory(plan.handle, rank, budget_bytes, C.byref(need), C.byref(budget)))
    return need.value, budget.value


def zero_bucket_range(plan: Plan, rank: int, bucket: int):
    b, e = C.c_uint64(), C.c_uint64()
    _check(_lib.zero_bucket_range(plan.handle, rank, bucket, C.byref(b), C.byref(e)))
    return b.value, e.value


def zero_reduce_scatter(plan: Plan, rank: int, grads, g_shard, stream=None):
    _check_step(plan, rank, grads, [("g_shard", g_shard)])
    _check(_lib.zero_reduce_scatter(plan.handle, rank, _ptr_array(grads, torch.bfloat16, "grads"),
                                    _dev(g_shard, torch.float32, "g_shard"), _stream(stream)))


def zero_adam_step(plan: Plan, rank: int, g_shard, master, m, v, param_out, hp, step: int, stream=None):
    _check_step(plan, rank, None, [("g_shard", g_shard), ("master", master), ("m", m), ("v", v)], param_out)
    a = _adam(hp)
    _check(_lib.zero_adam_step(plan.handle, rank, _dev(g_shard, torch.float32, "g_shard"),
                               _dev(master, torch.float32, "master"), _dev(m, torch.float32, "m"),
                               _dev(v, torch.float32, "v"), _dev(param_out, torch.bfloat16, "param_out"),
                               C.byref(a), step, _stream(stream)))


def zero_fused_step(plan: Plan, rank: int, grads, master, m, v, param_out, hp, step: int, stream=None):
    _check_step(plan, rank, grads, [("master", master), ("m", m), ("v", v)], param_out)
    a = _adam(hp)
    _check(_lib.zero_fused_step(plan.handle, rank, _ptr_array(grads, torch.bfloat16, "grads"),
                                _dev(master, torch.float32, "master"), _dev(m, torch.float32, "m"),
                                _dev(v, torch.float32, "v"), _dev(param_out, torch.bfloat16, "param_out"),
                                C.byref(a), step, _stream(stream)))


def _host(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError(f"{name} must be a CPU tensor in page-locked memory")
    if t.dtype != dtype or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous {dtype} tensor")
    if not t.is_pinned():
        raise ValueError(f"{name} must be page-locked (tensor.pin_memory())")
    return t.data_ptr()


def zero_fused_step_host(plan: Plan, rank: int, host_grads, master, m, v, host_param_out, hp, step: int, stream=None):
    """Fused step reading the ranks' gradients from page-locked host tensors and writing the
    bf16 parameters to a page-locked host tensor; master / m / v are CUDA tensors."""
    _check_step(plan, rank, host_grads, [("master", master), ("m", m), ("v", v)], host_param_out)
    a = _adam(hp)
    arr = (C.c_void_p * len(host_grads))(*[_host(g, torch.bfloat16, f"host_grads[{i}]")
                                          for i, g in enumerate(host_grads)])
    _check(_lib.zero_fused_step_host(plan.handle, rank, arr, _dev(master, torch.float32, "master"),
                                     _dev(m, torch.float32, "m"), _dev(v, torch.float32, "v"),
                                     _host(host_param_out, torch.bfloat16, "host_param_out"), C.byref(a), step,
                                     _stream(stream)))


def zero_fused_step_fp32_grads(plan: Plan, rank: int, grads, master, m, v, param_out, hp, step: int, stream=None):
    _check_step(plan, rank, grads, [("master", master), ("m", m), ("v", v)], param_out)
    a = _adam(hp)
    _check(_lib.zero_fused_step_fp32_grads(plan.handle, rank, _ptr_array(grads, torch.float32, "grads"),
                                           _dev(master, torch.float32, "master"), _dev(m, torch.float32, "m"),
                                           _dev(v, torch.float32, "v"), _dev(param_out, torch.bfloat16, "param_out"),
                                           C.byref(a), step, _stream(stream)))


def zero_fused_step_buckets(plan: Plan, rank: int, bucket_begin: int, bucket_end: int, grads, master, m, v,
                            param_out, hp, step: int, stream=None):
    _check_step(plan, rank, grads, [("master", master), ("m", m), ("v", v)], param_out)
    a = _adam(hp)
    _check(_lib.zero_fused_step_buckets(plan.handle, rank, bucket_begin, bucket_end,
                                        _ptr_array(grads, torch.bfloat16, "grads"),
                                        _dev(master, torch.float32, "master"), _dev(m, torch.float32, "m"),
                                        _dev(v, torch.float32, "v"), _dev(param_out, torch.bfloat16, "param_out"),
                                        C.byref(a), step, _stream(stream)))


def zero_allgather_params(plan: Plan, masters, full_param, stream=None):
    if len(masters) != plan.n_ranks:
        raise ValueError(f"masters holds {len(masters)} shards; the plan has {plan.n_ranks} ranks")
    for i, t in enumerate(masters):
        _need(t, plan.shard_elems, f"masters[{i}]")
    _need(full_param, plan.psi_padded, "full_param")
    _check(_lib.zero_allgather_params(plan.handle, _ptr_array(masters, torch.float32, "masters"),
                                      _dev(full_param, torch.bfloat16, "full_param"), _stream(stream)))


def ddp_allreduce(plan: Plan, grads, g_full, stream=None):
    _check_step(plan, ZERO_ALL_RANKS, grads, [("g_full", g_full)])
    _check(_lib.ddp_allreduce(plan.handle, _ptr_array(grads, torch.bfloat16, "grads"),
                              _dev(g_full, torch.float32, "g_full"), _stream(stream)))


def fsdp_gather_rows(w_shards, w_full, stream=None):
    n = len(w_shards)
    rs, k = _shards_shape(w_shards, "w_shards")
    if w_full.dim() != 2 or tuple(w_full.shape) != (n * rs, k):
        raise ValueError(f"w_full must be [{n * rs}, {k}] (got {tuple(w_full.shape)})")
    _check(_lib.fsdp_gather_rows(n, _ptr_array(w_shards, torch.bfloat16, "w_shards"), n * rs, k,
                                 _dev(w_full, torch.bfloat16, "w_full"), _stream(stream)))


def _forward_shapes(w_shards, A, Y, Y_bf16, scratch_w):
    n = len(w_shards)
    rs, k = _shards_shape(w_shards, "w_shards")
    if A.dim() != 2 or int(A.shape[1]) != k:
        raise ValueError(f"A must be [m_tokens, {k}] (got {tuple(A.shape)})")
    rows, m_tok = n * rs, int(A.shape[0])
    _need(Y, m_tok * rows, "Y")
    _need(Y_bf16, m_tok * rows, "Y_bf16")
    _need(scratch_w, rows * k, "scratch_w")
    return n, rows, k, m_tok


def fsdp_unit_forward(w_shards, A, Y, Y_bf16=None, scratch_w=None, stream=None):
    n, rows, k, m_tok = _forward_shapes(w_shards, A, Y, Y_bf16, scratch_w)
    _check(_lib.fsdp_unit_forward(n, _ptr_array(w_shards, torch.bfloat16, "w_shards"), rows, k,
                                  _dev(A, torch.bfloat16, "A"), m_tok, _dev(Y, torch.float32, "Y"),
                                  _dev(Y_bf16, torch.bfloat16, "Y_bf16"),
                                  _dev(scratch_w, torch.bfloat16, "scratch_w"), _stream(stream)))


def fsdp_transpose_cat(srcs, dst, stream=None):
    """dst [cols, n*rows] = the n row-major [rows, cols] bf16 sources transposed side by side."""
    rows, cols = _shards_shape(srcs, "srcs")
    _need(dst, len(srcs) * rows * cols, "dst")
    _check(_lib.fsdp_transpose_cat(len(srcs), _ptr_array(srcs, torch.bfloat16, "srcs"), rows, cols,
                                   _dev(dst, torch.bfloat16, "dst"), _stream(stream)))


def fsdp_unit_backward_workspace(n_ranks: int, rows_out: int, k_in: int, m_tokens: int) -> int:
    b = C.c_uint64()
    _check(_lib.fsdp_unit_backward_workspace(n_ranks, rows_out, k_in, m_tokens, C.byref(b)))
    return b.value


def fsdp_unit_backward(w_shards, A, dY, dX, dW, workspace=None, stream=None):
    """A, dY, dX: per-rank lists; dW: [rows_out, k_in] fp32; workspace: a uint8 CUDA tensor
    of at least fsdp_unit_backward_workspace(...) bytes (None where that is 0)."""
    n = len(w_shards)
    rs, k = _shards_shape(w_shards, "w_shards")
    rows = n * rs
    if not (len(A) == len(dY) == len(dX) == n):
        raise ValueError(f"A, dY and dX must hold one tensor per rank ({n})")
    m_tok, ka = _shards_shape(A, "A")
    if ka != k or _shards_shape(dY, "dY") != (m_tok, rows):
        raise ValueError(f"A must be [m_tokens, {k}] and dY [m_tokens, {rows}] per rank")
    for i, t in enumerate(dX):
        _need(t, m_tok * k, f"dX[{i}]")
    _need(dW, rows * k, "dW")
    _check(_lib.fsdp_unit_backward(
        n, _ptr_array(w_shards, torch.bfloat16, "w_shards"), rows, k, _ptr_array(A, torch.bfloat16, "A"),
        _ptr_array(dY, torch.bfloat16, "dY"), m_tok, _ptr_array(dX, torch.float32, "dX"),
        _dev(dW, torch.float32, "dW"), _dev(workspace, torch.uint8, "workspace"),
        0 if workspace is None else workspace.numel(), _stream(stream)))


def _unit_array(units, shapes_only=False):
    arr = (fsdp_unit_state * len(units))()
    for i, u in enumerate(units):
        rows, k = (int(u["w"].shape[0]), int(u["w"].shape[1])) if "w" in u else (int(u["rows_out"]), int(u["k_in"]))
        arr[i].rows_out, arr[i].k_in = rows, k
        if shapes_only:
            continue
        plan = u["plan"]
        arr[i].plan = plan.handle
        arr[i].w = _dev(u["w"], torch.bfloat16, f"units[{i}].w")
        for name in ("master", "m", "v"):
            _need(u[name], rows * k, f"units[{i}].{name}")
            setattr(arr[i], name, _dev(u[name], torch.float32, f"units[{i}].{name}"))
        nm = int(u["x"].shape[0]) if u["x"].dim() == 2 else -1
        if u["x"].dim() != 2 or int(u["x"].shape[1]) != k:
            raise ValueError(f"units[{i}].x must be [N*M, {k}] (got {tuple(u['x'].shape)})")
        if u["dy"].dim() != 2 or tuple(u["dy"].shape) != (nm, rows):
            raise ValueError(f"units[{i}].dy must be [{nm}, {rows}] (got {tuple(u['dy'].shape)})")
        _need(u.get("dw"), rows * k, f"units[{i}].dw")
        arr[i].x = _dev(u["x"], torch.bfloat16, f"units[{i}].x")
        arr[i].dy = _dev(u["dy"], torch.bfloat16, f"units[{i}].dy")
        arr[i].dw = _dev(u.get("dw"), torch.float32, f"units[{i}].dw")
    return arr


def fsdp_zero3_step_workspace(n_ranks: int, shapes, m_tokens: int, flags: int = 0) -> int:
    """Workspace bytes of fsdp_zero3_step for units of the given (rows_out, k_in) shapes."""
    arr = _unit_array([{"rows_out": r, "k_in": k} for r, k in shapes], shapes_only=True)
    b = C.c_uint64()
    _check(_lib.fsdp_zero3_step_workspace(n_ranks, len(arr), arr, m_tokens, flags, C.byref(b)))
    return b.value


def fsdp_zero3_step(units, m_tokens: int, hp, step: int, y_out=None, dx_out=None, flags: int = 0, workspace=None,
                    stream=None, prefetch_stream=None):
    """units: one dict per FSDP unit with plan, w [R, K] bf16 (the N row shards back to
    back), master / m / v fp32 [R*K], x [N*M, K] bf16, dy [N*M, R] bf16, dw [R, K] fp32."""
    if not units:
        raise ValueError("units is empty")
    n = units[0]["plan"].n_ranks
    arr = _unit_array(units)
    nm = n * m_tokens
    if int(units[0]["x"].shape[0]) != nm:
        raise ValueError(f"units[0].x must have N*M = {nm} rows")
    _need(y_out, nm * int(units[-1]["w"].shape[0]), "y_out")
    _need(dx_out, nm * int(units[0]["w"].shape[1]), "dx_out")
    a = _adam(hp)
    _check(_lib.fsdp_zero3_step(
        n, len(arr), arr, m_tokens, _dev(y_out, torch.bfloat16, "y_out"), _dev(dx_out, torch.bfloat16, "dx_out"),
        C.byref(a), step, flags, _dev(workspace, torch.uint8, "workspace"),
        0 if workspace is None else workspace.numel(), _stream(stream),
        None if prefetch_stream is None else _stream(prefetch_stream)))


def _weight_state(ws: fsdp_weight_state, w: dict, rows: int, cols: int, name: str):
    if tuple(w["w"].shape) != (rows, cols):
        raise ValueError(f"{name}.w must be [{rows}, {cols}] (got {tuple(w['w'].shape)})")
    ws.plan = w["plan"].handle
    ws.w = _dev(w["w"], torch.bfloat16, f"{name}.w")
    for k in ("master", "m", "v"):
        _need(w[k], rows * cols, f"{name}.{k}")
        setattr(ws, k, _dev(w[k], torch.float32, f"{name}.{k}"))


def _mlp_unit_array(units, nm=None):
    arr = (fsdp_mlp_unit_state * len(units))()
    for i, u in enumerate(units):
        d, f = int(u["d_model"]), int(u["d_ff"])
        arr[i].d_model, arr[i].d_ff = d, f
        if nm is None:
            continue
        _weight_state(arr[i].gate, u["gate"], f, d, f"units[{i}].gate")
        _weight_state(arr[i].up, u["up"], f, d, f"units[{i}].up")
        _weight_state(arr[i].down, u["down"], d, f, f"units[{i}].down")
        for k, cols in (("x", d), ("gu", 2 * f), ("h", f), ("dy", d), ("dh", f), ("dgu", 2 * f)):
            if u[k].dim() != 2 or tuple(u[k].shape) != (nm, cols):
                raise ValueError(f"units[{i}].{k} must be [{nm}, {cols}] (got {tuple(u[k].shape)})")
            setattr(arr[i], k, _dev(u[k], torch.bfloat16, f"units[{i}].{k}"))
        _need(u.get("dw_gu"), 2 * f * d, f"units[{i}].dw_gu")
        _need(u.get("dw_down"), d * f, f"units[{i}].dw_down")
        arr[i].dw_gu = _dev(u.get("dw_gu"), torch.float32, f"units[{i}].dw_gu")
        arr[i].dw_down = _dev(u.get("dw_down"), torch.float32, f"units[{i}].dw_down")
    return arr


def fsdp_zero3_mlp_step_workspace(n_ranks: int, shapes, m_tokens: int) -> int:
    """Workspace bytes of fsdp_zero3_mlp_step for MLP units of the given (d_model, d_ff)."""
    arr = _mlp_unit_array([{"d_model": d, "d_ff": f} for d, f in shapes])
    b = C.c_uint64()
    _check(_lib.fsdp_zero3_mlp_step_workspace(n_ranks, len(arr), arr, m_tokens, C.byref(b)))
    return b.value


def fsdp_zero3_mlp_step(units, m_tokens: int, hp, step: int, y_out=None, dx_out=None, workspace=None, stream=None,
                        flags: int = 0):
    """units: one dict per MLP unit with d_model, d_ff; gate / up / down as dicts of plan,
    w, master, m, v; and x, gu, h, dy, dh, dgu (bf16) and dw_gu, dw_down (fp32, or None
    when the optimizer is fused, the default)."""
    if not units:
        raise ValueError("units is empty")
    n = units[0]["gate"]["plan"].n_ranks
    nm = n * m_tokens
    arr = _mlp_unit_array(units, nm)
    _need(y_out, nm * int(units[-1]["d_model"]), "y_out")
    _need(dx_out, nm * int(units[0]["d_model"]), "dx_out")
    a = _adam(hp)
    _check(_lib.fsdp_zero3_mlp_step(
        n, len(arr), arr, m_tokens, _dev(y_out, torch.bfloat16, "y_out"), _dev(dx_out, torch.bfloat16, "dx_out"),
        C.byref(a), step, flags, _dev(workspace, torch.uint8, "workspace"),
        0 if workspace is None else workspace.numel(), _stream(stream)))


def fsdp_mlp_forward(gate_shards, up_shards, down_shards, X, H, Y, scratch_down=None, stream=None,
                     prefetch_stream=None):
    n = len(gate_shards)
    fs, d_model = _shards_shape(gate_shards, "gate_shards")
    d_ff = n * fs
    if len(up_shards) != n or _shards_shape(up_shards, "up_shards") != (fs, d_model):
        raise ValueError("up_shards must match gate_shards")
    ds, dff2 = _shards_shape(down_shards, "down_shards")
    if len(down_shards) != n or dff2 != d_ff or n * ds != d_model:
        raise ValueError(f"down_shards must be {n} shards of [{d_model // max(n, 1)}, {d_ff}]")
    if X.dim() != 2 or int(X.shape[1]) != d_model:
        raise ValueError(f"X must be [m_tokens, {d_model}] (got {tuple(X.shape)})")
    _need(H, int(X.shape[0]) * d_ff, "H")
    _need(Y, int(X.shape[0]) * d_model, "Y")
    _need(scratch_down, d_model * d_ff, "scratch_down")
    _check(_lib.fsdp_mlp_forward(
        n, _ptr_array(gate_shards, torch.bfloat16, "gate_shards"), _ptr_array(up_shards, torch.bfloat16, "up_shards"),
        _ptr_array(down_shards, torch.bfloat16, "down_shards"), d_model, d_ff, _dev(X, torch.bfloat16, "X"),
        int(X.shape[0]), _dev(H, torch.bfloat16, "H"), _dev(Y, torch.float32, "Y"),
        _dev(scratch_down, torch.bfloat16, "scratch_down"), _stream(stream),
        _stream(prefetch_stream) if prefetch_stream is not None else None))


def fsdp_unit_forward_static_scratch(w_shards, A, Y, Y_bf16=None, stream=None):
    """fsdp_unit_forward with the gathered W in the library's own 16 MiB device array
    (for callers that cannot allocate); no scratch argument."""
    n, rows, k, m_tok = _forward_shapes(w_shards, A, Y, Y_bf16, None)
    _check(_lib.fsdp_unit_forward_static_scratch(
        n, _ptr_array(w_shards, torch.bfloat16, "w_shards"), rows, k, _dev(A, torch.bfloat16, "A"),
        m_tok, _dev(Y, torch.float32, "Y"), _dev(Y_bf16, torch.bfloat16, "Y_bf16"), _stream(stream)))


def zero_device_status(stream=None):
    _check(_lib.zero_device_status(_stream(stream)))


def zero_selftest_bounded_wait(timeout_ms: int, stream=None):
    _check(_lib.zero_selftest_bounded_wait(timeout_ms, _stream(stream)))


def zero_set_fused_kernel(which: int):
    _check(_lib.zero_set_fused_kernel(which))


def zero_set_gemm_kernel(which: int):
    _check(_lib.zero_set_gemm_kernel(which))


def zero_version() -> int:
    return _lib.zero_version()


def zero_last_error() -> str:
    return _lib.zero_last_error().decode(errors="replace")


def library():
    """The loaded ctypes library (for tests that call the C ABI directly)."""
    return _lib
