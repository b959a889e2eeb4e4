"""Thin Python binding of libmfsdp.so (the C ABI declared in include/mfsdp.h).

Argument marshalling only: every step of the owner-local optimizer step runs in
the library's CUDA kernels.  Device buffers are torch tensors (PyTorch supplies
device memory and streams); the library never allocates.  Importing this
module raises if the library has not been built -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import List, Optional, Sequence, Tuple

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libmfsdp.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libmfsdp.so is not built ({_LIB_PATH}); run __graft_entry__.build()")
_lib = ctypes.CDLL(_LIB_PATH)

OK = 0
ERR_INVALID_ARG = -1
ERR_MISALIGNED = -2
ERR_OVERLAP = -3
ERR_OUT_OF_BOUNDS = -4
ERR_UNSUPPORTED_DTYPE = -5
ERR_UNSUPPORTED_SHAPE = -6
ERR_WORKSPACE_TOO_SMALL = -7
ERR_CUDA = -8
ERR_DEVICE_TIMEOUT = -9
ERR_IO = -10
ERR_FORMAT = -11

DTYPE_F32 = 0
DTYPE_BF16 = 1
KIND_MATRIX = 0
KIND_TAIL = 1

PHASE_MOMENTUM = 1
PHASE_NEWTON_SCHULZ = 2

EXPORTED = ("mfsdp_plan_owners", "mfsdp_muon_workspace_bytes", "mfsdp_muon_owner_step", "mfsdp_muon_owner_step_phases",
            "mfsdp_muon_device_status", "mfsdp_muon_workspace_layout", "mfsdp_adamw_tail_step",
            "mfsdp_status_string", "mfsdp_version", "mfsdp_muon_owner_step_static_scratch",
            "mfsdp_muon_step_flops", "mfsdp_muon_owner_step_host", "mfsdp_muon_owner_step_apply",
            "mfsdp_model_layout", "mfsdp_placement_segments", "mfsdp_segment_copy", "mfsdp_test_inject_stall",
            "mfsdp_host_step_groups", "mfsdp_muon_static_scratch_status", "mfsdp_checkpoint_bytes",
            "mfsdp_checkpoint_write", "mfsdp_checkpoint_read_header", "mfsdp_checkpoint_read",
            "mfsdp_muon_gram_space_layout")

SEGMENT_REDUCE = 0
SEGMENT_GATHER = 1

SCALE_NONE = 0      # scale = 1
SCALE_MUON = 1      # scale = sqrt(max(1, rows/cols))
SCALE_RMS = 2       # scale = 0.2 * sqrt(max(rows, cols))

STATIC_SCRATCH_BYTES = 64 << 20


class CParam(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("kind", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class MatrixShard(ctypes.Structure):
    _fields_ = [("param_id", ctypes.c_int32), ("owner", ctypes.c_int32), ("offset", ctypes.c_int64),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("transposed", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("cost", ctypes.c_uint64)]

    def as_dict(self) -> dict:
        return dict(param_id=self.param_id, owner=self.owner, offset=self.offset, rows=self.rows,
                    cols=self.cols, transposed=self.transposed, cost=self.cost)


class TailShard(ctypes.Structure):
    _fields_ = [("param_id", ctypes.c_int32), ("owner", ctypes.c_int32), ("offset", ctypes.c_int64),
                ("numel", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return dict(param_id=self.param_id, owner=self.owner, offset=self.offset, numel=self.numel)


_i32, _i64, _u64, _d, _vp, _sz = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double,
                                  ctypes.c_void_p, ctypes.c_size_t)
_lib.mfsdp_plan_owners.argtypes = [ctypes.POINTER(CParam), _i32, _i32, _i32, _i64, ctypes.POINTER(MatrixShard),
                                   ctypes.POINTER(_i32), ctypes.POINTER(TailShard), ctypes.POINTER(_i32),
                                   ctypes.POINTER(_i64), ctypes.POINTER(_i64)]
_lib.mfsdp_plan_owners.restype = ctypes.c_int
_lib.mfsdp_muon_workspace_bytes.argtypes = [ctypes.POINTER(MatrixShard), _i32]
_lib.mfsdp_muon_workspace_bytes.restype = _sz
_lib.mfsdp_muon_workspace_layout.argtypes = [ctypes.POINTER(MatrixShard), _i32, ctypes.POINTER(_i64)]
_lib.mfsdp_muon_workspace_layout.restype = ctypes.c_int
_lib.mfsdp_muon_gram_space_layout.argtypes = [ctypes.POINTER(MatrixShard), _i32, _i32, ctypes.POINTER(_i64)]
_lib.mfsdp_muon_gram_space_layout.restype = ctypes.c_int
_STEP_ARGS = [ctypes.POINTER(MatrixShard), _i32, _vp, _i32, _vp, _vp, _i32, _i64, _d, _i32, _i32, _d, _d, _d, _d,
              _vp, _sz, _vp]
_lib.mfsdp_muon_owner_step.argtypes = _STEP_ARGS
_lib.mfsdp_muon_owner_step.restype = ctypes.c_int
_lib.mfsdp_muon_owner_step_phases.argtypes = _STEP_ARGS + [_i32]
_lib.mfsdp_muon_owner_step_phases.restype = ctypes.c_int
_lib.mfsdp_muon_owner_step_host.argtypes = [ctypes.POINTER(MatrixShard), _i32, _vp, _vp, _i32, _vp, _vp, _vp, _i32,
                                            _i64, _d, _i32, _i32, _d, _d, _d, _d, _vp, _sz, _i32, _vp]
_lib.mfsdp_muon_owner_step_host.restype = ctypes.c_int
_lib.mfsdp_host_step_groups.argtypes = [ctypes.POINTER(MatrixShard), _i32, _i32, _i32, _i32,
                                        ctypes.POINTER(_i32)]
_lib.mfsdp_host_step_groups.restype = _i32
_lib.mfsdp_muon_owner_step_apply.argtypes = [ctypes.POINTER(MatrixShard), _i32, _vp, _i32, _vp, _vp, _i32, _vp, _i32,
                                             _i64, _d, _i32, _i32, _d, _d, _d, _d, _d, _d, _i32, _vp, _sz, _vp]
_lib.mfsdp_muon_owner_step_apply.restype = ctypes.c_int
_lib.mfsdp_muon_owner_step_static_scratch.argtypes = _STEP_ARGS[:15] + [_vp]
_lib.mfsdp_muon_owner_step_static_scratch.restype = ctypes.c_int
_lib.mfsdp_muon_step_flops.argtypes = [ctypes.POINTER(MatrixShard), _i32, _i32, ctypes.POINTER(_u64),
                                       ctypes.POINTER(_u64)]
_lib.mfsdp_muon_step_flops.restype = ctypes.c_int
_lib.mfsdp_muon_device_status.argtypes = [_vp, _vp, ctypes.POINTER(_i32)]
_lib.mfsdp_muon_device_status.restype = ctypes.c_int
_lib.mfsdp_muon_static_scratch_status.argtypes = [_vp, ctypes.POINTER(_i32)]
_lib.mfsdp_muon_static_scratch_status.restype = ctypes.c_int
_lib.mfsdp_test_inject_stall.argtypes = [_i32]
_lib.mfsdp_test_inject_stall.restype = ctypes.c_int
_lib.mfsdp_adamw_tail_step.argtypes = [_vp, _vp, _vp, _vp, _i64, _d, _d, _d, _d, _d, _i64, _vp]
_lib.mfsdp_adamw_tail_step.restype = ctypes.c_int
_lib.mfsdp_status_string.argtypes = [ctypes.c_int]
_lib.mfsdp_status_string.restype = ctypes.c_char_p
_lib.mfsdp_version.argtypes = []
_lib.mfsdp_version.restype = ctypes.c_char_p


class MfsdpError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


def status_string(status: int) -> str:
    return _lib.mfsdp_status_string(int(status)).decode()


def version() -> str:
    return _lib.mfsdp_version().decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise MfsdpError(status, what)


@dataclasses.dataclass
class Plan:
    matrix_shards: List[MatrixShard]
    tail_shards: List[TailShard]
    rank_matrix_elems: List[int]
    rank_tail_elems: List[int]

    def rank_matrices(self, r: int) -> List[MatrixShard]:
        return [s for s in self.matrix_shards if s.owner == r]

    def rank_tails(self, r: int) -> List[TailShard]:
        return [s for s in self.tail_shards if s.owner == r]


def plan_owners(params: Sequence[Tuple[int, int, int]], world: int, ns_steps: int = 5,
                align_elems: int = 128) -> Plan:
    """Balance-aware owner plan: params are (rows, cols, kind) in declaration order."""
    n = len(params)
    arr = (CParam * max(n, 1))()
    for i, (r, c, k) in enumerate(params):
        arr[i].rows, arr[i].cols, arr[i].kind = int(r), int(c), int(k)
    nm = sum(1 for p in params if p[2] == KIND_MATRIX)
    nt = n - nm
    out_m = (MatrixShard * max(nm, 1))()
    out_t = (TailShard * max(nt, 1))()
    cm, ct = _i32(0), _i32(0)
    world_i = int(world)
    rme = (_i64 * max(world_i, 1))()
    rte = (_i64 * max(world_i, 1))()
    _check(_lib.mfsdp_plan_owners(arr, n, world_i, int(ns_steps), int(align_elems), out_m, ctypes.byref(cm), out_t,
                                  ctypes.byref(ct), rme, rte), "plan_owners")
    return Plan([out_m[i] for i in range(cm.value)], [out_t[i] for i in range(ct.value)],
                list(rme[:world_i]), list(rte[:world_i]))


def _shard_array(shards: Sequence[MatrixShard]):
    arr = (MatrixShard * max(len(shards), 1))()
    for i, s in enumerate(shards):
        arr[i] = s
    return arr


class Placement(ctypes.Structure):
    _fields_ = [("param_id", ctypes.c_int32), ("owner", ctypes.c_int32), ("offset", ctypes.c_int64),
                ("numel", ctypes.c_int64)]


class Segment(ctypes.Structure):
    _fields_ = [("src_offset", ctypes.c_int64), ("dst_offset", ctypes.c_int64), ("numel", ctypes.c_int64),
                ("src_index", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return dict(src_index=self.src_index, src_offset=self.src_offset, dst_offset=self.dst_offset,
                    numel=self.numel)


def placements(plan: "Plan") -> Tuple[List[Placement], List[Placement]]:
    """The plan's matrix shards and tail shards as placements (param, owner, offset, numel)."""
    def mk(pid, owner, off, n):
        p = Placement()
        p.param_id, p.owner, p.offset, p.numel = pid, owner, off, n
        return p
    return ([mk(s.param_id, s.owner, s.offset, s.rows * s.cols) for s in plan.matrix_shards],
            [mk(s.param_id, s.owner, s.offset, s.numel) for s in plan.tail_shards])


def model_layout(params: Sequence[Tuple[int, int, int]], align_elems: int = 128) -> Tuple[List[int], int]:
    """Offsets of the parameters in the unsharded flat layout, and its extent."""
    n = len(params)
    arr = (CParam * max(n, 1))()
    for i, (r, c, k) in enumerate(params):
        arr[i].rows, arr[i].cols, arr[i].kind = int(r), int(c), int(k)
    offs = (ctypes.c_int64 * max(n, 1))()
    total = ctypes.c_int64(0)
    _check(_lib.mfsdp_model_layout(arr, n, int(align_elems), offs, ctypes.byref(total)), "model_layout")
    return list(offs[:n]), int(total.value)


def model_placements(params: Sequence[Tuple[int, int, int]], align_elems: int = 128) -> List[Placement]:
    """Every parameter in the unsharded layout, as placements with owner 0."""
    offs, _ = model_layout(params, align_elems)
    out = []
    for i, (r, c, _) in enumerate(params):
        p = Placement()
        p.param_id, p.owner, p.offset, p.numel = i, 0, offs[i], r * c
        out.append(p)
    return out


def placement_segments(src: Sequence[Placement], dst: Sequence[Placement], dst_owner: int) -> List[Segment]:
    """Segments that fill dst_owner's buffer of `dst` from `src` (see include/mfsdp.h)."""
    a = (Placement * max(len(src), 1))(*src)
    b = (Placement * max(len(dst), 1))(*dst)
    out = (Segment * max(len(dst), 1))()
    n = ctypes.c_int32(0)
    _check(_lib.mfsdp_placement_segments(a, len(src), b, len(dst), int(dst_owner), out, ctypes.byref(n)),
           "placement_segments")
    return [out[i] for i in range(n.value)]


def segment_copy(srcs, segs: Sequence[Segment], mode: int, dst, stream=None) -> None:
    """REDUCE (sum of all sources in order) or GATHER the segments into dst."""
    n = len(srcs)
    ptrs = (ctypes.c_void_p * max(n, 1))(*[_ptr(t) for t in srcs])
    sizes = (ctypes.c_int64 * max(n, 1))(*[int(t.numel()) for t in srcs])
    arr = (Segment * max(len(segs), 1))(*segs)
    _check(_lib.mfsdp_segment_copy(ptrs, sizes, n, _dtype_code(srcs[0]), arr, len(segs), int(mode), _ptr(dst),
                                   _dtype_code(dst), int(dst.numel()), _stream(stream)), "segment_copy")


def make_shard(offset: int, rows: int, cols: int, param_id: int = 0, owner: int = 0) -> MatrixShard:
    s = MatrixShard()
    s.param_id, s.owner, s.offset, s.rows, s.cols = param_id, owner, offset, rows, cols
    s.transposed = int(rows > cols)
    return s


def muon_workspace_bytes(shards: Sequence[MatrixShard]) -> int:
    return int(_lib.mfsdp_muon_workspace_bytes(_shard_array(shards), len(shards)))


def muon_workspace_layout(shards: Sequence[MatrixShard]) -> List[Tuple[int, ...]]:
    out = (_i64 * max(8 * len(shards), 1))()
    _check(_lib.mfsdp_muon_workspace_layout(_shard_array(shards), len(shards), out), "muon_workspace_layout")
    return [tuple(out[8 * i: 8 * i + 8]) for i in range(len(shards))]


def muon_gram_space_layout(shards: Sequence[MatrixShard], ns_steps: int = 5) -> List[Tuple[int, ...]]:
    """Per shard (1 if the Gram-space form runs else 0, offset of C, of Q_even,
    of Q_odd) for ns_steps (see include/mfsdp.h)."""
    out = (_i64 * max(4 * len(shards), 1))()
    _check(_lib.mfsdp_muon_gram_space_layout(_shard_array(shards), len(shards), int(ns_steps), out),
           "muon_gram_space_layout")
    return [tuple(out[4 * i: 4 * i + 4]) for i in range(len(shards))]


def muon_step_flops(shards: Sequence[MatrixShard], ns_steps: int = 5) -> Tuple[int, int]:
    """(dense, executed) FLOPs of one owner step (see include/mfsdp.h)."""
    dn, ex = _u64(0), _u64(0)
    _check(_lib.mfsdp_muon_step_flops(_shard_array(shards), len(shards), int(ns_steps), ctypes.byref(dn),
                                      ctypes.byref(ex)), "muon_step_flops")
    return int(dn.value), int(ex.value)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    return 99   # rejected by the library as UNSUPPORTED_DTYPE


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    return int(stream) if isinstance(stream, int) else int(stream.cuda_stream)


def muon_owner_step(shards: Sequence[MatrixShard], grad, momentum, update, workspace, *, beta: float = 0.95,
                    nesterov: bool = False, ns_steps: int = 5, coeffs=(3.4445, -4.7750, 2.0315),
                    eps: float = 1e-7, numel: Optional[int] = None, stream=None,
                    phases: int = PHASE_MOMENTUM | PHASE_NEWTON_SCHULZ) -> None:
    """One owner-local Muon step over the shards of one rank (see include/mfsdp.h).

    grad: flat fp32/bf16 CUDA tensor; momentum: flat fp32; update: flat fp32/bf16;
    workspace: CUDA uint8 tensor of at least muon_workspace_bytes(shards) bytes.
    phases: both (default, mfsdp_muon_owner_step) or one of PHASE_MOMENTUM /
    PHASE_NEWTON_SCHULZ (mfsdp_muon_owner_step_phases)."""
    arr = _shard_array(shards)
    n = int(numel if numel is not None else grad.numel())
    a, b, c = coeffs
    args = (arr, len(shards), _ptr(grad), _dtype_code(grad), _ptr(momentum), _ptr(update), _dtype_code(update), n,
            float(beta), int(bool(nesterov)), int(ns_steps), float(a), float(b), float(c), float(eps),
            _ptr(workspace), int(workspace.numel() if workspace is not None else 0), _stream(stream))
    if phases == PHASE_MOMENTUM | PHASE_NEWTON_SCHULZ:
        _check(_lib.mfsdp_muon_owner_step(*args), "muon_owner_step")
    else:
        _check(_lib.mfsdp_muon_owner_step_phases(*args, int(phases)), "muon_owner_step_phases")


def muon_owner_step_apply(shards: Sequence[MatrixShard], grad, momentum, update, weights, workspace, *, lr: float,
                          weight_decay: float = 0.0, scale_mode: int = SCALE_MUON, beta: float = 0.95,
                          nesterov: bool = False, ns_steps: int = 5, coeffs=(3.4445, -4.7750, 2.0315),
                          eps: float = 1e-7, numel: Optional[int] = None, stream=None) -> None:
    """The owner step, then W <- W*(1 - lr*wd) - lr*scale*O fused into the last
    epilogue (see include/mfsdp.h).  update may be None."""
    arr = _shard_array(shards)
    n = int(numel if numel is not None else grad.numel())
    a, b, c = coeffs
    _check(_lib.mfsdp_muon_owner_step_apply(arr, len(shards), _ptr(grad), _dtype_code(grad), _ptr(momentum),
                                            _ptr(update), _dtype_code(update) if update is not None else DTYPE_BF16,
                                            _ptr(weights), _dtype_code(weights), n, float(beta), int(bool(nesterov)),
                                            int(ns_steps), float(a), float(b), float(c), float(eps), float(lr),
                                            float(weight_decay), int(scale_mode), _ptr(workspace),
                                            int(workspace.numel() if workspace is not None else 0), _stream(stream)),
           "muon_owner_step_apply")


def muon_owner_step_host(shards: Sequence[MatrixShard], grad_host, grad_dev, momentum, update_dev, update_host,
                         workspace, *, groups: int = 0, beta: float = 0.95, nesterov: bool = False,
                         ns_steps: int = 5, coeffs=(3.4445, -4.7750, 2.0315), eps: float = 1e-7,
                         numel: Optional[int] = None, stream=None) -> None:
    """The owner step with the gradient read from and the update written to pinned
    host tensors, the copies of each shard group overlapped with the compute of
    its neighbours (see include/mfsdp.h).  grad_dev/update_dev are device staging
    tensors of the same length.  groups = 0: the count host_step_groups gives."""
    arr = _shard_array(shards)
    n = int(numel if numel is not None else grad_dev.numel())
    a, b, c = coeffs
    _check(_lib.mfsdp_muon_owner_step_host(arr, len(shards), _ptr(grad_host), _ptr(grad_dev), _dtype_code(grad_dev),
                                           _ptr(momentum), _ptr(update_dev), _ptr(update_host), _dtype_code(update_dev),
                                           n, float(beta), int(bool(nesterov)), int(ns_steps), float(a), float(b),
                                           float(c), float(eps), _ptr(workspace),
                                           int(workspace.numel() if workspace is not None else 0), int(groups),
                                           _stream(stream)),
           "muon_owner_step_host")


def host_step_groups(shards: Sequence[MatrixShard], grad_dtype=None, update_dtype=None,
                     groups: int = 0) -> Tuple[int, List[int]]:
    """(number of groups, each shard's group) of the host-buffer step for
    `groups` (0 = the library's choice); host only.  The dtypes are torch
    dtypes, bf16 gradient and update by default."""
    import torch
    g = torch.bfloat16 if grad_dtype is None else grad_dtype
    u = torch.bfloat16 if update_dtype is None else update_dtype
    code = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}
    out = (_i32 * max(len(shards), 1))()
    ng = int(_lib.mfsdp_host_step_groups(_shard_array(shards), len(shards), code.get(g, 99), code.get(u, 99),
                                         int(groups), out))
    return ng, [int(out[i]) for i in range(len(shards))] if ng else []


def muon_owner_step_static_scratch(shards: Sequence[MatrixShard], grad, momentum, update, *, beta: float = 0.95,
                                   nesterov: bool = False, ns_steps: int = 5, coeffs=(3.4445, -4.7750, 2.0315),
                                   eps: float = 1e-7, numel: Optional[int] = None, stream=None) -> None:
    """The owner step for callers that cannot allocate device memory: no
    workspace argument; the library's fixed STATIC_SCRATCH_BYTES device array
    serves as scratch (see include/mfsdp.h).  Calls that overlap on the GPU race."""
    arr = _shard_array(shards)
    n = int(numel if numel is not None else grad.numel())
    a, b, c = coeffs
    _check(_lib.mfsdp_muon_owner_step_static_scratch(arr, len(shards), _ptr(grad), _dtype_code(grad), _ptr(momentum),
                                                     _ptr(update), _dtype_code(update), n, float(beta),
                                                     int(bool(nesterov)), int(ns_steps), float(a), float(b), float(c),
                                                     float(eps), _stream(stream)),
           "muon_owner_step_static_scratch")


def test_inject_stall(tile: int) -> None:
    """Testing only: the next Newton-Schulz launch's tile `tile` waits for a
    dependency that is never satisfied, so its bounded wait runs out (see
    include/mfsdp.h)."""
    _check(_lib.mfsdp_test_inject_stall(int(tile)), "test_inject_stall")


def muon_device_status(workspace, stream=None) -> Tuple[int, int]:
    detail = _i32(0)
    st = _lib.mfsdp_muon_device_status(_ptr(workspace), _stream(stream), ctypes.byref(detail))
    return st, detail.value


def muon_static_scratch_status(stream=None) -> Tuple[int, int]:
    """(status, raw word) of the last static-scratch step on the current device
    (synchronises the stream; see include/mfsdp.h)."""
    detail = _i32(0)
    st = _lib.mfsdp_muon_static_scratch_status(_stream(stream), ctypes.byref(detail))
    return st, detail.value


def adamw_tail_step(p, g, m, v, *, lr: float, beta1: float, beta2: float, eps: float, wd: float, step: int,
                    stream=None) -> None:
    """Fused AdamW over one rank's packed fp32 tail (see include/mfsdp.h)."""
    n = int(p.numel())
    _check(_lib.mfsdp_adamw_tail_step(_ptr(p), _ptr(g), _ptr(m), _ptr(v), n, float(lr), float(beta1), float(beta2),
                                      float(eps), float(wd), int(step), _stream(stream)), "adamw_tail_step")


_lib.mfsdp_model_layout.argtypes = [ctypes.POINTER(CParam), _i32, _i64, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]
_lib.mfsdp_model_layout.restype = ctypes.c_int
_lib.mfsdp_placement_segments.argtypes = [ctypes.POINTER(Placement), _i32, ctypes.POINTER(Placement), _i32, _i32,
                                          ctypes.POINTER(Segment), ctypes.POINTER(_i32)]
_lib.mfsdp_placement_segments.restype = ctypes.c_int
_lib.mfsdp_segment_copy.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(_i64), _i32, _i32,
                                    ctypes.POINTER(Segment), _i32, _i32, _vp, _i32, _i64, _vp]
_lib.mfsdp_segment_copy.restype = ctypes.c_int


class CheckpointHeader(ctypes.Structure):
    _fields_ = [("world", ctypes.c_int32), ("rank", ctypes.c_int32), ("ns_steps", ctypes.c_int32),
                ("n_matrix", ctypes.c_int32), ("n_tail", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("align_elems", ctypes.c_int64), ("matrix_elems", ctypes.c_int64), ("tail_elems", ctypes.c_int64),
                ("adam_step", ctypes.c_int64)]


_lib.mfsdp_checkpoint_bytes.argtypes = [ctypes.POINTER(CheckpointHeader)]
_lib.mfsdp_checkpoint_bytes.restype = _sz
_lib.mfsdp_checkpoint_write.argtypes = [ctypes.c_char_p, ctypes.POINTER(CheckpointHeader), ctypes.POINTER(MatrixShard),
                                        ctypes.POINTER(TailShard), _vp, _vp, _vp, _vp]
_lib.mfsdp_checkpoint_write.restype = ctypes.c_int
_lib.mfsdp_checkpoint_read_header.argtypes = [ctypes.c_char_p, ctypes.POINTER(CheckpointHeader)]
_lib.mfsdp_checkpoint_read_header.restype = ctypes.c_int
_lib.mfsdp_checkpoint_read.argtypes = [ctypes.c_char_p, ctypes.POINTER(CheckpointHeader), ctypes.POINTER(MatrixShard),
                                       _i32, ctypes.POINTER(TailShard), _i32, _vp, _i64, _vp, _vp, _vp, _i64]
_lib.mfsdp_checkpoint_read.restype = ctypes.c_int


@dataclasses.dataclass
class Checkpoint:
    """One rank's owner-shard checkpoint: its header, tables and host buffers
    (NumPy float32 arrays)."""
    header: CheckpointHeader
    matrix_shards: List[MatrixShard]
    tail_shards: List[TailShard]
    momentum: "object"
    tail_p: "object"
    tail_m: "object"
    tail_v: "object"


def _host_f32(x, n: int):
    """A C-contiguous float32 NumPy copy of a tensor or array of n elements."""
    import numpy as np
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if a.size != n:
        raise ValueError(f"buffer has {a.size} elements, the header says {n}")
    return a


def checkpoint_save(path: str, world: int, rank: int, ns_steps: int, align_elems: int,
                    matrix_shards: Sequence[MatrixShard], tail_shards: Sequence[TailShard], momentum, tail_p, tail_m,
                    tail_v, adam_step: int) -> None:
    """Writes one rank's state (momentum and the AdamW tail's p, m, v, as
    tensors or arrays; copied to host memory here) with its tables (see
    include/mfsdp.h)."""
    h = CheckpointHeader()
    h.world, h.rank, h.ns_steps = int(world), int(rank), int(ns_steps)
    h.n_matrix, h.n_tail, h.align_elems = len(matrix_shards), len(tail_shards), int(align_elems)
    h.matrix_elems = int(momentum.numel() if hasattr(momentum, "numel") and callable(momentum.numel)
                         else len(momentum))
    h.tail_elems = int(tail_p.numel() if hasattr(tail_p, "numel") and callable(tail_p.numel) else len(tail_p))
    h.adam_step = int(adam_step)
    bufs = [_host_f32(momentum, h.matrix_elems)] + [_host_f32(t, h.tail_elems) for t in (tail_p, tail_m, tail_v)]
    marr = _shard_array(matrix_shards)
    tarr = (TailShard * max(len(tail_shards), 1))(*tail_shards)
    _check(_lib.mfsdp_checkpoint_write(os.fsencode(path), ctypes.byref(h), marr, tarr,
                                       *[b.ctypes.data for b in bufs]), "checkpoint_write")


def checkpoint_load(path: str) -> Checkpoint:
    """Reads one rank's checkpoint into host memory (see include/mfsdp.h)."""
    import numpy as np
    h = CheckpointHeader()
    _check(_lib.mfsdp_checkpoint_read_header(os.fsencode(path), ctypes.byref(h)), "checkpoint_read_header")
    marr = (MatrixShard * max(h.n_matrix, 1))()
    tarr = (TailShard * max(h.n_tail, 1))()
    mom = np.empty(h.matrix_elems, np.float32)
    tail = [np.empty(h.tail_elems, np.float32) for _ in range(3)]
    _check(_lib.mfsdp_checkpoint_read(os.fsencode(path), ctypes.byref(h), marr, h.n_matrix, tarr, h.n_tail,
                                      mom.ctypes.data, h.matrix_elems, *[t.ctypes.data for t in tail], h.tail_elems),
           "checkpoint_read")
    return Checkpoint(h, [marr[i] for i in range(h.n_matrix)], [tarr[i] for i in range(h.n_tail)], mom, *tail)


def library_path() -> str:
    """Path of the loaded libmfsdp.so."""
    return _LIB_PATH


def raw_lib() -> ctypes.CDLL:
    """The loaded library, for callers that marshal raw pointers themselves."""
    return _lib
