"""Python binding of libmla_decode.so (include/mla_decode.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  Tensors must already live on the current CUDA
device; outputs, metadata and scratch are torch allocations owned by the
caller.  There is no CPU path: if the library is missing or no GPU is present
the calls raise.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libmla_decode.so"
D_QK, D_V, BLOCK_SIZE = 576, 512, 64

_lib = None


class MLAError(RuntimeError):
    pass


def load_library():
    """Loads libmla_decode.so (built by mla_decode_attention_03_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not LIB_PATH.exists():
        raise MLAError(f"{LIB_PATH} is missing: build it with "
                       "`python -m mla_decode_attention_03_gb300.build` (needs nvcc for sm_103a)")
    lib = ctypes.CDLL(str(LIB_PATH))
    P, I, I64, SZ, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_status_string.argtypes = [ctypes.c_int32]
    lib.mla_num_parts.restype = I
    lib.mla_num_parts.argtypes = [I, I, I, I]
    lib.mla_metadata_ints.restype = SZ
    lib.mla_metadata_ints.argtypes = [I]
    lib.mla_workspace_bytes.restype = SZ
    lib.mla_workspace_bytes.argtypes = [I, I, I, I]
    lib.mla_get_metadata.restype = ctypes.c_int32
    lib.mla_get_metadata.argtypes = [P, I, I, P, P, P, P]
    for name in ("mla_decode_with_kvcache", "mla_decode_splitkv", "mla_selftest_wait_timeout"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int32
        fn.argtypes = [P, I, I, I, I, P, I64, I, I, I, P, I, P, I, P, I, P, F, I, P, P, P, SZ, P, P]
    lib.mla_combine_splits.restype = ctypes.c_int32
    lib.mla_combine_splits.argtypes = [P, I, I, I, P, I, P, P, P]
    lib.mla_write_cache.restype = ctypes.c_int32
    lib.mla_write_cache.argtypes = [P, I64, P, I64, P, I64, P, I64, I, I, P, P]
    lib.mla_copy_blocks.restype = ctypes.c_int32
    lib.mla_copy_blocks.argtypes = [P, I, P, I64, I64, I, I, P, P]
    lib.mla_host_pipeline_create.restype = ctypes.c_int32
    lib.mla_host_pipeline_create.argtypes = [ctypes.POINTER(P)]
    lib.mla_host_pipeline_destroy.restype = ctypes.c_int32
    lib.mla_host_pipeline_destroy.argtypes = [P]
    lib.mla_host_chunks.restype = I
    lib.mla_host_chunks.argtypes = [P, I, I, P]
    lib.mla_host_scratch_bytes.restype = SZ
    lib.mla_host_scratch_bytes.argtypes = [I, I, I, I, I]
    lib.mla_decode_host.restype = ctypes.c_int32
    lib.mla_decode_host.argtypes = [P, P, I, I, I, I, P, I64, I, I, I, P, I, P, I, I, F, I, P, P, I, P, SZ, P, P]
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().mla_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != 0:
        raise MLAError(f"{what}: {status_string(code)} ({code})")


def _stream_handle() -> int:
    return torch.cuda.current_stream().cuda_stream


def num_parts(s_q: int, h_q: int, h_kv: int = 1, device=None) -> int:
    dev = torch.cuda.current_device() if device is None else torch.device(device).index or 0
    n = load_library().mla_num_parts(s_q, h_q, h_kv, dev)
    if n < 0:
        _check(n, "mla_num_parts")
    return n


def workspace_bytes(b: int, s_q: int, h_q: int, parts: int) -> int:
    return int(load_library().mla_workspace_bytes(b, s_q, h_q, parts))


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word for the calls below."""
    return torch.zeros(1, dtype=torch.int32, device=device or torch.cuda.current_device())


def check_status(status: torch.Tensor):
    """Synchronises on the status word and raises if a kernel reported an error."""
    code = int(status.item())
    if code != 0:
        raise MLAError(f"device reported {status_string(code)} ({code})")


def get_mla_metadata(cache_seqlens: torch.Tensor, parts: int, status: torch.Tensor | None = None):
    """Split-KV schedule: returns (metadata int32[parts, 8], num_splits int32[b+1])."""
    assert cache_seqlens.is_cuda and cache_seqlens.dtype == torch.int32 and cache_seqlens.dim() == 1
    sl = cache_seqlens.contiguous()
    b = sl.shape[0]
    meta = torch.empty((parts, 8), dtype=torch.int32, device=sl.device)
    nsplit = torch.empty((b + 1,), dtype=torch.int32, device=sl.device)
    if status is None:
        status = new_status(sl.device)
    _check(load_library().mla_get_metadata(sl.data_ptr(), b, parts, meta.data_ptr(), nsplit.data_ptr(),
                                           status.data_ptr(), _stream_handle()), "mla_get_metadata")
    return meta, nsplit


def entry_stride(kcache: torch.Tensor) -> int:
    """Elements between consecutive entries of a [num_blocks, 64, h_kv, 576]
    cache view (576 when dense, 640 for the 256-byte aligned layout)."""
    nb, bs, h_kv, d = kcache.shape
    st = kcache.stride()
    es = st[2] if h_kv > 1 else st[1]
    if st[3] != 1 or st[1] != h_kv * es or st[0] != bs * st[1]:
        raise MLAError(f"kcache layout not supported: shape {tuple(kcache.shape)}, strides {st}")
    return es


def _check_io(q, block_table, cache_seqlens, out, lse, dv=D_V):
    """Shapes, types and layouts of the per-sequence arrays against q
    [b, s_q, h_q, d]: the library reads and writes exactly these extents, so a
    smaller tensor must be refused here, before its pointer is handed over."""
    if q.dim() != 4:
        raise MLAError(f"q must be [b, s_q, h_q, d], got shape {tuple(q.shape)}")
    b, s_q, h_q, _ = q.shape
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != b:
        raise MLAError(f"block_table must be int32 [{b}, max_blocks], got {block_table.dtype} "
                       f"{tuple(block_table.shape)}")
    if cache_seqlens.dtype != torch.int32 or tuple(cache_seqlens.shape) != (b,):
        raise MLAError(f"cache_seqlens must be int32 [{b}], got {cache_seqlens.dtype} {tuple(cache_seqlens.shape)}")
    for name, t, shape, dtype in (("out", out, (b, s_q, h_q, dv), torch.bfloat16),
                                  ("lse", lse, (b, h_q, s_q), torch.float32)):
        if t is None:
            continue
        if tuple(t.shape) != shape or t.dtype != dtype or not t.is_contiguous():
            raise MLAError(f"{name} must be a contiguous {dtype} tensor of shape {shape}, got {t.dtype} "
                           f"{tuple(t.shape)}{'' if t.is_contiguous() else ' (not contiguous)'}")
        if t.device != q.device:
            raise MLAError(f"{name} must be on {q.device}")


def mla_decode_with_kvcache(q: torch.Tensor, kcache: torch.Tensor, block_table: torch.Tensor,
                            cache_seqlens: torch.Tensor, metadata: torch.Tensor,
                            num_splits: torch.Tensor, softmax_scale: float, causal: bool = False,
                            dv: int = D_V, out: torch.Tensor | None = None,
                            lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                            status: torch.Tensor | None = None, combine: bool = True):
    """MLA decode: returns (out bf16[b, s_q, h_q, 512], lse fp32[b, h_q, s_q]).

    combine=False runs only the split-KV decode kernel (mla_decode_splitkv);
    combine_splits() must then follow on the same stream."""
    if not (q.is_cuda and kcache.is_cuda):
        raise MLAError("q and kcache must be CUDA tensors")
    if q.dtype != torch.bfloat16 or kcache.dtype != torch.bfloat16:
        raise MLAError("q and kcache must be bfloat16")
    if not q.is_contiguous():
        raise MLAError("q must be contiguous")
    _check_io(q, block_table, cache_seqlens, out, lse, dv)
    b, s_q, h_q, d = q.shape
    nb, bs, h_kv, dk = kcache.shape
    stride = entry_stride(kcache)
    bt = block_table.contiguous()
    sl = cache_seqlens.contiguous()
    if not (bt.device == sl.device == kcache.device == q.device):
        raise MLAError("q, kcache, block_table and cache_seqlens must be on one device")
    if tuple(num_splits.shape) != (b + 1,) or metadata.dim() != 2 or metadata.shape[1] != 8:
        raise MLAError("metadata / num_splits do not come from get_mla_metadata for this batch")
    parts = metadata.shape[0]
    dev = q.device
    if out is None:
        out = torch.empty((b, s_q, h_q, dv), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((b, h_q, s_q), dtype=torch.float32, device=dev)
    need = workspace_bytes(b, s_q, h_q, parts)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    if status is None:
        status = new_status(dev)
    lib = load_library()
    fn = lib.mla_decode_with_kvcache if combine else lib.mla_decode_splitkv
    rc = fn(
        q.data_ptr(), b, s_q, h_q, d, kcache.data_ptr(), nb, bs, h_kv, stride, bt.data_ptr(),
        bt.shape[1], sl.data_ptr(), dv, metadata.data_ptr(), parts, num_splits.data_ptr(),
        float(softmax_scale), int(bool(causal)), out.data_ptr(), lse.data_ptr(),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), status.data_ptr(),
        _stream_handle())
    _check(rc, "mla_decode_with_kvcache" if combine else "mla_decode_splitkv")
    return out, lse


def combine_splits(num_splits: torch.Tensor, workspace: torch.Tensor, parts: int, out: torch.Tensor,
                   lse: torch.Tensor):
    """The merge half of mla_decode_with_kvcache (mla_combine_splits)."""
    if out.dim() != 4 or out.shape[3] != D_V or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise MLAError(f"out must be a contiguous bfloat16 [b, s_q, h_q, {D_V}] tensor")
    b, s_q, h_q, _ = out.shape
    if (tuple(lse.shape) != (b, h_q, s_q) or lse.dtype != torch.float32 or not lse.is_contiguous()
            or lse.device != out.device):
        raise MLAError(f"lse must be a contiguous float32 [{b}, {h_q}, {s_q}] tensor on {out.device}")
    if tuple(num_splits.shape) != (b + 1,):
        raise MLAError(f"num_splits must have {b + 1} entries")
    if workspace.numel() * workspace.element_size() < workspace_bytes(b, s_q, h_q, parts):
        raise MLAError("workspace smaller than mla_workspace_bytes for this shape")
    _check(load_library().mla_combine_splits(num_splits.data_ptr(), b, s_q, h_q, workspace.data_ptr(),
                                             parts, out.data_ptr(), lse.data_ptr(), _stream_handle()),
           "mla_combine_splits")
    return out, lse


def write_cache(kv_c: torch.Tensor, k_pe: torch.Tensor, slot_mapping: torch.Tensor, kcache: torch.Tensor,
                status: torch.Tensor | None = None):
    """New tokens into the paged cache: entry slot_mapping[t] <- [kv_c[t], k_pe[t]]
    (mla_write_cache).  kcache is the [num_blocks, 64, 1, 576] view of the cache."""
    if kv_c.dtype != torch.bfloat16 or k_pe.dtype != torch.bfloat16 or kcache.dtype != torch.bfloat16:
        raise MLAError("kv_c, k_pe and kcache must be bfloat16")
    if kv_c.stride(-1) != 1 or k_pe.stride(-1) != 1:
        raise MLAError("kv_c and k_pe rows must be contiguous")
    if kv_c.shape[-1] != 512 or k_pe.shape[-1] != 64 or kv_c.dim() != 2 or k_pe.dim() != 2:
        raise MLAError("kv_c must be [T, 512] and k_pe [T, 64]")
    if kv_c.shape[0] != k_pe.shape[0] or slot_mapping.numel() != kv_c.shape[0]:
        raise MLAError("kv_c, k_pe and slot_mapping must have one row per token")
    if kv_c.device != kcache.device or k_pe.device != kcache.device:
        raise MLAError("kv_c, k_pe and kcache must be on one device")
    sm = slot_mapping.to(device=kcache.device, dtype=torch.int64).contiguous()
    nb, bs, h_kv, _ = kcache.shape
    if h_kv != 1:
        raise MLAError("MLA caches have one latent head")
    if status is None:
        status = new_status(kcache.device)
    _check(load_library().mla_write_cache(kv_c.data_ptr(), kv_c.stride(0), k_pe.data_ptr(), k_pe.stride(0),
                                          sm.data_ptr(), sm.numel(), kcache.data_ptr(), nb, bs,
                                          entry_stride(kcache), status.data_ptr(), _stream_handle()),
           "mla_write_cache")
    return kcache


def copy_blocks(kcaches: list, block_mapping: torch.Tensor, status: torch.Tensor | None = None):
    """copy_blocks_mla: for every layer cache and (src, dst) pair, page dst <- page src."""
    if not kcaches:
        return kcaches
    nb, bs, h_kv, _ = kcaches[0].shape
    stride = entry_stride(kcaches[0])
    for c in kcaches:
        if c.dtype != torch.bfloat16 or c.device != kcaches[0].device:
            raise MLAError("layer caches must be bfloat16 tensors on one device")
        if c.shape != kcaches[0].shape or entry_stride(c) != stride:
            raise MLAError("all layer caches must share one shape and entry stride")
    dev = kcaches[0].device
    ptrs = torch.tensor([c.data_ptr() for c in kcaches], dtype=torch.int64, device=dev)
    bm = block_mapping.to(device=dev, dtype=torch.int64).contiguous()
    if bm.dim() != 2 or bm.shape[1] != 2:
        raise MLAError(f"block_mapping must be [num_pairs, 2], got {tuple(bm.shape)}")
    if status is None:
        status = new_status(dev)
    _check(load_library().mla_copy_blocks(ptrs.data_ptr(), len(kcaches), bm.data_ptr(), bm.shape[0], nb, bs,
                                          stride, status.data_ptr(), _stream_handle()), "mla_copy_blocks")
    return kcaches


class MLADecoder:
    """Holds the per-step schedule, scratch and status word for one decode shape.

    plan(cache_seqlens) once per decode step (the schedule is shared by all
    layers), then __call__ once per layer."""

    def __init__(self, b: int, s_q: int, h_q: int, h_kv: int = 1, device=None, parts: int | None = None):
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.b, self.s_q, self.h_q, self.h_kv = b, s_q, h_q, h_kv
        self.parts = parts if parts is not None else num_parts(s_q, h_q, h_kv, self.device)
        self.workspace = torch.empty((workspace_bytes(b, s_q, h_q, self.parts),), dtype=torch.uint8,
                                     device=self.device)
        self.status = new_status(self.device)
        self.metadata = None
        self.num_splits = None

    def plan(self, cache_seqlens: torch.Tensor):
        self.metadata, self.num_splits = get_mla_metadata(cache_seqlens, self.parts, self.status)
        return self

    def __call__(self, q, kcache, block_table, cache_seqlens, softmax_scale, causal=False, out=None, lse=None):
        return mla_decode_with_kvcache(q, kcache, block_table, cache_seqlens, self.metadata,
                                       self.num_splits, softmax_scale, causal, out=out, lse=lse,
                                       workspace=self.workspace, status=self.status)


HOST_MAX_CHUNKS = 8  # MLA_HOST_MAX_CHUNKS


def host_chunks(cache_seqlens: torch.Tensor, chunks: int = 0) -> list:
    """The cut of a batch into runs of consecutive sequences that the
    host-buffer decode makes (mla_host_chunks): sequence bounds [0, ..., b]."""
    sl = cache_seqlens.to(torch.int32).contiguous()
    assert sl.device.type == "cpu" and sl.dim() == 1
    bounds = (ctypes.c_int32 * (HOST_MAX_CHUNKS + 1))()
    n = load_library().mla_host_chunks(sl.data_ptr(), sl.shape[0], int(chunks), ctypes.addressof(bounds))
    if n < 0:
        _check(n, "mla_host_chunks")
    return list(bounds[: n + 1])


class HostDecoder:
    """Decode from host tensors (mla_decode_host): q, block_table and
    cache_seqlens are CPU tensors (pinned for the copies to overlap), out and
    lse come back in CPU tensors; the KV cache stays on the device.  The batch
    is cut into runs of sequences whose copies in and out overlap the decode
    of the neighbouring runs.  Holds the pipeline's streams and events and the
    device staging scratch for batches up to (b, s_q, h_q, max_blocks_per_seq).

    The call returns once the work is enqueued on the current stream: keep the
    host tensors alive and unchanged, and read out/lse only after
    torch.cuda.current_stream().synchronize() (or check_status(self.status))."""

    def __init__(self, b: int, s_q: int, h_q: int, max_blocks_per_seq: int, h_kv: int = 1, device=None,
                 parts: int | None = None):
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.b, self.s_q, self.h_q, self.h_kv, self.max_blocks = b, s_q, h_q, h_kv, max_blocks_per_seq
        self.parts = parts if parts is not None else num_parts(s_q, h_q, h_kv, self.device)
        lib = load_library()
        self._handle = None
        with torch.cuda.device(self.device):
            h = ctypes.c_void_p()
            _check(lib.mla_host_pipeline_create(ctypes.byref(h)), "mla_host_pipeline_create")
            self._handle = h
        n = lib.mla_host_scratch_bytes(b, s_q, h_q, max_blocks_per_seq, self.parts)
        if n == 0:
            raise MLAError("mla_host_scratch_bytes: invalid shape")
        # zeroed once: no run can ever see stale schedule words, whatever was in the memory before
        self.scratch = torch.zeros((n,), dtype=torch.uint8, device=self.device)
        self.status = new_status(self.device)

    def __call__(self, q, kcache, block_table, cache_seqlens, softmax_scale, causal=False, out=None, lse=None,
                 chunks: int = 0):
        if self._handle is None:
            raise MLAError("HostDecoder is closed")
        for name, t in (("q", q), ("block_table", block_table), ("cache_seqlens", cache_seqlens)):
            if t.device.type != "cpu" or not t.is_contiguous():
                raise MLAError(f"{name} must be a contiguous CPU tensor")
        if q.dtype != torch.bfloat16 or kcache.dtype != torch.bfloat16 or not kcache.is_cuda:
            raise MLAError("q must be bfloat16 on the host and kcache bfloat16 on the device")
        if block_table.dtype != torch.int32 or cache_seqlens.dtype != torch.int32:
            raise MLAError("block_table and cache_seqlens must be int32")
        _check_io(q, block_table, cache_seqlens, out, lse)
        b, s_q, h_q, d = q.shape
        if b > self.b or s_q != self.s_q or h_q != self.h_q or block_table.shape[1] > self.max_blocks:
            raise MLAError(f"shape {tuple(q.shape)} / max_blocks {block_table.shape[1]} outside the decoder's "
                           f"({self.b}, {self.s_q}, {self.h_q}) / {self.max_blocks}")
        nb, bs, h_kv, dk = kcache.shape
        stride = entry_stride(kcache)
        if out is None:
            out = torch.empty((b, s_q, h_q, D_V), dtype=torch.bfloat16, pin_memory=True)
        if lse is None:
            lse = torch.empty((b, h_q, s_q), dtype=torch.float32, pin_memory=True)
        if out.device.type != "cpu" or lse.device.type != "cpu" or not (out.is_contiguous() and lse.is_contiguous()):
            raise MLAError("out and lse must be contiguous CPU tensors")
        with torch.cuda.device(self.device):
            rc = load_library().mla_decode_host(
                self._handle, q.data_ptr(), b, s_q, h_q, d, kcache.data_ptr(), nb, bs, h_kv, stride,
                block_table.data_ptr(), block_table.shape[1], cache_seqlens.data_ptr(), D_V, self.parts,
                float(softmax_scale), int(bool(causal)), out.data_ptr(), lse.data_ptr(), int(chunks),
                self.scratch.data_ptr(), self.scratch.numel(), self.status.data_ptr(), _stream_handle())
        _check(rc, "mla_decode_host")
        return out, lse

    def close(self):
        if self._handle is not None:
            h, self._handle = self._handle, None
            _check(load_library().mla_host_pipeline_destroy(h), "mla_host_pipeline_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
