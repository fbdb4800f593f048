"""GB300-native batched beam-search step, KV-cache reorder and blockwise verify.

A thin ctypes binding over ``libvbs.so`` (declared in ``include/vbs.h``): every
function here only marshals torch tensors into pointers, sizes and the current
CUDA stream; all of the work runs in the library's CUDA kernels.  There is no
fallback: if the library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["BeamSearch", "PagedKV", "kv_reorder", "bpd_propose", "bpd_verify", "VbsError", "lib",
           "LP_GNMT", "LP_POWER", "ES_FALSE", "ES_TRUE", "ES_NEVER", "F32", "BF16", "BPD_EXACT", "BPD_TOPK",
           "BPD_DISTANCE", "gather_shard_partials"]

F32, BF16 = 0, 1
LP_GNMT, LP_POWER = 0, 1
BPD_EXACT, BPD_TOPK, BPD_DISTANCE = 0, 1, 2
ES_FALSE, ES_TRUE, ES_NEVER = 0, 1, 2
OK, EINVAL, ECUDA, ENOMEM, ESTATE, EALIGN, ETIMEOUT, EINPUT, ESCRATCH, EBOUNDS = 0, -1, -2, -3, -4, -5, -6, -7, -8, -9

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libvbs.so")
CHECKED_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libvbs_checked.so")

_c_int, _c_i64, _c_f, _vp = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
_pp = ctypes.POINTER(ctypes.c_void_p)

# name -> (restype, argtypes); mirrors include/vbs.h
SIGNATURES = {
    "vbs_strerror": (ctypes.c_char_p, [_c_int]),
    "vbs_version": (_c_int, []),
    "bs_init": (_c_int, [_pp, _c_int, _c_int, _c_int, _c_int, ctypes.c_double, _c_int, _c_int, _c_int, _c_int, _c_int,
                         _c_int, _vp]),
    "bs_reset": (_c_int, [_vp, _vp, _vp]),
    "bs_step": (_c_int, [_vp, _vp, _c_i64, _vp, _vp, _vp, _vp, _vp]),
    "bs_finalize": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "bs_finalize_n": (_c_int, [_vp, _vp, _vp, _c_int, _vp, _vp, _vp]),
    "bs_finished": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "bs_seqs": (_c_int, [_vp, _pp]),
    "bs_steps": (_c_int, [_vp, ctypes.POINTER(_c_int)]),
    "bs_status": (_c_int, [_vp]),
    "bs_destroy": (_c_int, [_vp]),
    "bs_expand_static": (_c_int, [_vp, _c_i64, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp, _vp, _vp]),
    "kv_reorder": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _vp]),
    "vbs_stateless_status": (_c_int, [_vp]),
    "kv_paged_init": (_c_int, [_pp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp]),
    "kv_paged_prefill": (_c_int, [_vp, _c_int]),
    "kv_paged_prepare": (_c_int, [_vp, _c_int]),
    "kv_paged_reorder": (_c_int, [_vp, _vp, _c_int]),
    "bs_step_two_pass": (_c_int, [_vp, _vp, _c_i64, _vp, _vp, _vp, _vp, _vp]),
    "bs_shard_partial_bytes": (_c_int, [_vp, _vp]),
    "bs_step_shard": (_c_int, [_vp, _vp, _c_i64, _c_int, _c_int, _vp, _vp]),
    "bs_step_merge_shards": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _vp, _vp, _vp]),
    "bs_step_paged": (_c_int, [_vp, _vp, _c_i64, _vp, _vp, _vp, _vp, _vp, _vp, _c_int]),
    "kv_paged_copy": (_c_int, [_vp]),
    "kv_paged_table": (_c_int, [_vp, _pp, ctypes.POINTER(_c_int)]),
    "kv_paged_counts": (_c_int, [_vp, _vp, _vp]),
    "kv_paged_copy_table": (_c_int, [_vp, _vp]),
    "kv_paged_save": (_c_int, [_vp]),
    "kv_paged_cow_slots": (_c_int, [_vp, ctypes.POINTER(_c_i64)]),
    "kv_paged_restore": (_c_int, [_vp]),
    "kv_paged_status": (_c_int, [_vp]),
    "kv_paged_destroy": (_c_int, [_vp]),
    "bpd_propose": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp]),
    "bpd_verify": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp]),
    "bpd_verify_approx": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp,
                                   _vp]),
    "vbs_peak_copy": (_c_int, [_vp, _vp, _c_i64, _c_int, _vp]),
    "vbs_peak_read": (_c_int, [_vp, _c_i64, _c_int, _c_int, _vp, _vp]),
    "vbs_checked_record": (_c_int, [ctypes.POINTER(_c_int), ctypes.POINTER(_c_int), ctypes.POINTER(_c_i64)]),
}

_LIB = None


class VbsError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        msg = lib().vbs_strerror(status).decode() if _LIB is not None else str(status)
        super().__init__(f"{what}: {msg} ({status})" if what else f"{msg} ({status})")
        self.status = status


def lib():
    """Load libvbs.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m verify_bs_step_gb300._build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _LIB = L
    return _LIB


def load_checked():
    """The checked build (libvbs_checked.so: device bounds checks on), loaded with the same
    signatures; swap it in with `use_library(...)`."""
    if not os.path.exists(CHECKED_LIB_PATH):
        raise RuntimeError(f"{CHECKED_LIB_PATH} is missing: build it with `python -m verify_bs_step_gb300._build`")
    L = ctypes.CDLL(CHECKED_LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype, fn.argtypes = res, args
    return L


def use_library(L):
    """Make every call of this module go to library L (returns the one it replaces)."""
    global _LIB
    old, _LIB = _LIB, L
    return old


def checked_record():
    """(checked build?, site, index) of the first failed device bounds check since the last call."""
    c, site, idx = _c_int(), _c_int(), _c_i64()
    _check(lib().vbs_checked_record(ctypes.byref(c), ctypes.byref(site), ctypes.byref(idx)), "vbs_checked_record")
    return bool(c.value), site.value, idx.value


def _check(st: int, what: str):
    if st != OK:
        raise VbsError(st, what)


def _dev_ptr(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return _vp(t.data_ptr())


def _stream(device=None):
    return _vp(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(dt) -> int:
    if dt == torch.bfloat16:
        return BF16
    if dt == torch.float32:
        return F32
    raise ValueError(f"logits dtype must be bfloat16 or float32, got {dt}")


class BeamSearch:
    """Batched beam search over `batch` sentences x W beams (libvbs bs_*).

    Holds the decode's device buffers (scores [R] fp32, seqs [R, max_len+1]
    int32, beam_idx [R], tokens [R], an all-done flag) so steps allocate nothing.
    All work goes on the stream that is current at construction.
    """

    def __init__(self, batch: int, W: int, V: int, *, eos: int = -1, alpha: float = 1.0,
                 early_stopping: int = ES_FALSE, lp_kind: int = LP_GNMT, max_len: int = 64, bos: int = 0,
                 pad: int = -1, dtype=torch.bfloat16, device="cuda"):
        self.batch, self.W, self.V, self.max_len = batch, W, V, max_len
        self.R = batch * W
        self.device = torch.device(device)
        self.dtype = dtype
        self._stream_obj = torch.cuda.current_stream(self.device)
        self.stream = _vp(self._stream_obj.cuda_stream)
        ctx = _vp()
        _check(lib().bs_init(ctypes.byref(ctx), batch, W, V, eos, alpha, early_stopping, lp_kind, max_len, bos,
                             pad, _dtype_code(dtype), self.stream), "bs_init")
        self.ctx = ctx
        dev = self.device
        self.scores = torch.empty(self.R, dtype=torch.float32, device=dev)
        self.seqs = torch.empty(self.R, max_len + 1, dtype=torch.int32, device=dev)
        self.beam_idx = torch.empty(self.R, dtype=torch.int32, device=dev)
        self.tokens = torch.empty(self.R, dtype=torch.int32, device=dev)
        self.all_done = torch.zeros(1, dtype=torch.int32, device=dev)
        self.reset()

    def reset(self):
        _check(lib().bs_reset(self.ctx, _vp(self.scores.data_ptr()), _vp(self.seqs.data_ptr())), "bs_reset")

    def step(self, logits: torch.Tensor):
        """One step on logits [R, V] (unit stride along V); returns (beam_idx, tokens, scores) views."""
        if logits.dim() != 2 or logits.shape[0] != self.R or logits.shape[1] != self.V or logits.stride(1) != 1:
            raise ValueError(f"logits must be [{self.R}, {self.V}] with unit stride along V")
        if logits.dtype != self.dtype:
            raise ValueError(f"logits must be {self.dtype}")
        _check(lib().bs_step(self.ctx, _dev_ptr(logits, "logits"), logits.stride(0), _vp(self.scores.data_ptr()),
                             _vp(self.seqs.data_ptr()), _vp(self.beam_idx.data_ptr()),
                             _vp(self.tokens.data_ptr()), _vp(self.all_done.data_ptr())), "bs_step")
        return self.beam_idx, self.tokens, self.scores

    def step_two_pass(self, logits: torch.Tensor):
        """step() through the two-pass coarse-selection ablation (reads the logits twice)."""
        if logits.dim() != 2 or logits.shape[0] != self.R or logits.shape[1] != self.V or logits.stride(1) != 1:
            raise ValueError(f"logits must be [{self.R}, {self.V}] with unit stride along V")
        if logits.dtype != self.dtype:
            raise ValueError(f"logits must be {self.dtype}")
        _check(lib().bs_step_two_pass(self.ctx, _dev_ptr(logits, "logits"), logits.stride(0),
                                      _vp(self.scores.data_ptr()), _vp(self.seqs.data_ptr()),
                                      _vp(self.beam_idx.data_ptr()), _vp(self.tokens.data_ptr()),
                                      _vp(self.all_done.data_ptr())), "bs_step_two_pass")
        return self.beam_idx, self.tokens, self.scores

    def shard_partial(self, logits_shard: torch.Tensor, v0: int) -> torch.Tensor:
        """The partial of vocabulary columns [v0, v0 + Vs) of this step's logits (a [R, Vs] view,
        unit stride along V): a uint8 device tensor of bs_shard_partial_bytes()."""
        if logits_shard.dim() != 2 or logits_shard.shape[0] != self.R or logits_shard.stride(1) != 1:
            raise ValueError(f"logits_shard must be [{self.R}, Vs] with unit stride along V")
        if logits_shard.dtype != self.dtype:
            raise ValueError(f"logits must be {self.dtype}")
        n = ctypes.c_int64()
        _check(lib().bs_shard_partial_bytes(self.ctx, ctypes.byref(n)), "bs_shard_partial_bytes")
        out = torch.empty(n.value, dtype=torch.uint8, device=self.device)
        _check(lib().bs_step_shard(self.ctx, _dev_ptr(logits_shard, "logits"), logits_shard.stride(0), v0,
                                   logits_shard.shape[1], _vp(self.scores.data_ptr()), _vp(out.data_ptr())),
               "bs_step_shard")
        return out

    def merge_shards(self, partials: torch.Tensor):
        """Finish the step from the shards' partials ([n_shards, bytes] uint8, contiguous, device);
        returns (beam_idx, tokens, scores) views like step()."""
        if partials.dim() != 2 or not partials.is_contiguous() or partials.dtype != torch.uint8:
            raise ValueError("partials must be a contiguous [n_shards, bytes] uint8 tensor")
        _check(lib().bs_step_merge_shards(self.ctx, partials.shape[0], _dev_ptr(partials, "partials"),
                                          _vp(self.scores.data_ptr()), _vp(self.seqs.data_ptr()),
                                          _vp(self.beam_idx.data_ptr()), _vp(self.tokens.data_ptr()),
                                          _vp(self.all_done.data_ptr())), "bs_step_merge_shards")
        return self.beam_idx, self.tokens, self.scores

    def step_paged(self, logits: torch.Tensor, kv: "PagedKV", t_valid: int):
        """step() plus the table remap of kv.reorder(beam_idx, t_valid); the copy-on-write
        runs at kv.copy().  Returns (beam_idx, tokens, scores) views."""
        if logits.dim() != 2 or logits.shape[0] != self.R or logits.shape[1] != self.V or logits.stride(1) != 1:
            raise ValueError(f"logits must be [{self.R}, {self.V}] with unit stride along V")
        if logits.dtype != self.dtype:
            raise ValueError(f"logits must be {self.dtype}")
        _check(lib().bs_step_paged(self.ctx, _dev_ptr(logits, "logits"), logits.stride(0),
                                   _vp(self.scores.data_ptr()), _vp(self.seqs.data_ptr()),
                                   _vp(self.beam_idx.data_ptr()), _vp(self.tokens.data_ptr()),
                                   _vp(self.all_done.data_ptr()), kv.ctx, t_valid), "bs_step_paged")
        return self.beam_idx, self.tokens, self.scores

    def finalize(self, n_return: int = 1):
        """(out_seqs [batch * n, max_len+1] int32, out_len [batch * n] int32, out_score [batch * n] fp32):
        the best n_return hypotheses of each sentence, best first (sentence b's j-th in row b * n + j)."""
        rows = self.batch * n_return
        out = torch.empty(rows, self.max_len + 1, dtype=torch.int32, device=self.device)
        out_len = torch.empty(rows, dtype=torch.int32, device=self.device)
        out_score = torch.empty(rows, dtype=torch.float32, device=self.device)
        if n_return == 1:
            _check(lib().bs_finalize(self.ctx, _vp(self.scores.data_ptr()), _vp(self.seqs.data_ptr()),
                                     _vp(out.data_ptr()), _vp(out_len.data_ptr()), _vp(out_score.data_ptr())),
                   "bs_finalize")
        else:
            _check(lib().bs_finalize_n(self.ctx, _vp(self.scores.data_ptr()), _vp(self.seqs.data_ptr()), n_return,
                                       _vp(out.data_ptr()), _vp(out_len.data_ptr()), _vp(out_score.data_ptr())),
                   "bs_finalize_n")
        return out, out_len, out_score

    def finished(self):
        """The finished sets: dict of count [B], ns [R] fp64, len [R], serial [R], tokens [R, max_len+1], done [B]."""
        d = self.device
        f = {"count": torch.empty(self.batch, dtype=torch.int32, device=d),
             "ns": torch.empty(self.R, dtype=torch.float64, device=d),
             "len": torch.empty(self.R, dtype=torch.int32, device=d),
             "serial": torch.empty(self.R, dtype=torch.int32, device=d),
             "tokens": torch.empty(self.R, self.max_len + 1, dtype=torch.int32, device=d),
             "done": torch.empty(self.batch, dtype=torch.int32, device=d)}
        _check(lib().bs_finished(self.ctx, *[_vp(f[k].data_ptr()) for k in
                                             ("count", "ns", "len", "serial", "tokens", "done")]), "bs_finished")
        return f

    def steps(self) -> int:
        n = _c_int()
        _check(lib().bs_steps(self.ctx, ctypes.byref(n)), "bs_steps")
        return n.value

    def status(self) -> int:
        """Synchronise and return the device status word (0 = OK)."""
        return lib().bs_status(self.ctx)

    def close(self):
        if getattr(self, "ctx", None) is not None and self.ctx.value:
            lib().bs_destroy(self.ctx)
            self.ctx = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def bs_expand_static(logits: torch.Tensor, scores_in: torch.Tensor, W: int, scores_out: torch.Tensor | None = None,
                     beam_idx: torch.Tensor | None = None, tokens: torch.Tensor | None = None):
    """One beam expansion (no end-of-sequence token) through the allocation-free entry point.

    logits: CUDA [batch*W, V] (row stride may exceed V), float32 or bfloat16; scores_in: float32
    [batch*W].  Returns (beam_idx, tokens, scores_out).  The library itself allocates nothing;
    the output tensors this wrapper creates when none are given are torch's.
    """
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be [rows, V] with unit column stride")
    R, V = logits.shape
    if W < 1 or R % W:
        raise ValueError("rows must be a multiple of W")
    dev = logits.device
    if scores_out is None:
        scores_out = torch.empty(R, dtype=torch.float32, device=dev)
    if beam_idx is None:
        beam_idx = torch.empty(R, dtype=torch.int32, device=dev)
    if tokens is None:
        tokens = torch.empty(R, dtype=torch.int32, device=dev)
    # the kernels read and write R contiguous entries of each on the logits' device
    for name, t in (("scores_in", scores_in), ("scores_out", scores_out), ("beam_idx", beam_idx),
                    ("tokens", tokens)):
        if t.numel() != R or not t.is_contiguous() or t.device != dev:
            raise ValueError(f"{name} must be a contiguous tensor of {R} entries on {dev}")
    _check(lib().bs_expand_static(_dev_ptr(logits, "logits"), logits.stride(0), R // W, W, V,
                                  _dtype_code(logits.dtype), _dev_ptr(scores_in, "scores_in", torch.float32),
                                  _dev_ptr(scores_out, "scores_out", torch.float32),
                                  _dev_ptr(beam_idx, "beam_idx", torch.int32),
                                  _dev_ptr(tokens, "tokens", torch.int32), _stream(dev)),
           "bs_expand_static")
    return beam_idx, tokens, scores_out


def peak_copy(src: torch.Tensor, dst: torch.Tensor, grid: int):
    """Copy src's bytes into dst with the library's vector-copy kernel (`grid` CTAs)."""
    if not (src.is_contiguous() and dst.is_contiguous()) or src.nbytes != dst.nbytes:
        raise ValueError("src and dst must be contiguous and of equal size")
    _check(lib().vbs_peak_copy(_dev_ptr(src, "src"), _dev_ptr(dst, "dst"), src.nbytes, grid, _stream(src.device)),
           "vbs_peak_copy")


def peak_read(src: torch.Tensor, grid: int, mode: int, sink: torch.Tensor):
    """Read src's bytes with the library's read-only streaming kernel (mode 0: vector loads,
    mode 1: bulk-copy ring); sink is an int32 tensor of at least `grid` entries."""
    if not src.is_contiguous() or sink.numel() < grid or sink.dtype != torch.int32:
        raise ValueError("src must be contiguous; sink int32 with >= grid entries")
    _check(lib().vbs_peak_read(_dev_ptr(src, "src"), src.nbytes, grid, mode, _dev_ptr(sink, "sink"),
                               _stream(src.device)), "vbs_peak_read")


class _KvDesc(ctypes.Structure):
    _fields_ = [("layers", _c_int), ("heads", _c_int), ("head_dim", _c_int), ("t_max", _c_int),
                ("elem_bytes", _c_int)]


def kv_reorder(src: torch.Tensor, dst: torch.Tensor, beam_idx: torch.Tensor, t_valid: int):
    """dst[:, :, r, :, :t_valid] = src[:, :, beam_idx[r], :, :t_valid] for beam_idx[r] >= 0.

    src, dst: contiguous [L, 2, rows, H, T_max, D] CUDA tensors; beam_idx: int32 [rows].
    """
    if src.shape != dst.shape or src.dim() != 6 or src.shape[1] != 2:
        raise ValueError("src and dst must be [L, 2, rows, H, T_max, D]")
    if not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("src and dst must be contiguous")
    L, _, rows, H, T, D = src.shape
    desc = _KvDesc(L, H, D, T, src.element_size())
    _check(lib().kv_reorder(ctypes.byref(desc), _dev_ptr(src, "src"), _dev_ptr(dst, "dst"),
                            _dev_ptr(beam_idx, "beam_idx", torch.int32), rows, t_valid, _stream(src.device)),
           "kv_reorder")


class PagedKV:
    """Paged KV cache with copy-on-write (libvbs kv_paged_*).

    The pool is a [batch * blocks_per_sentence, L, 2, H, block, D] tensor; the
    library owns the block table, the reference counts and the free stacks.
    """

    def __init__(self, batch: int, W: int, L: int, H: int, D: int, *, blocks_per_sentence: int,
                 max_blocks: int, block: int = 16, dtype=torch.bfloat16, device="cuda", pool=None):
        self.batch, self.W, self.R = batch, W, batch * W
        self.L, self.H, self.D, self.block = L, H, D, block
        self.S, self.max_blocks = blocks_per_sentence, max_blocks
        self.device = torch.device(device)
        if pool is None:
            pool = torch.zeros(batch * blocks_per_sentence, L, 2, H, block, D, dtype=dtype, device=self.device)
        self.pool = pool
        self.stream = _vp(torch.cuda.current_stream(self.device).cuda_stream)
        desc = _KvDesc(L, H, D, max_blocks * block, pool.element_size())
        ctx = _vp()
        _check(lib().kv_paged_init(ctypes.byref(ctx), ctypes.byref(desc), batch, W, blocks_per_sentence, block,
                                   max_blocks, _dev_ptr(pool, "pool"), self.stream), "kv_paged_init")
        self.ctx = ctx
        ptr = _vp()
        mb = _c_int()
        _check(lib().kv_paged_table(self.ctx, ctypes.byref(ptr), ctypes.byref(mb)), "kv_paged_table")
        self._table_ptr = ptr.value

    def prefill(self, P: int):
        _check(lib().kv_paged_prefill(self.ctx, P), "kv_paged_prefill")

    def prepare(self, t_write: int):
        _check(lib().kv_paged_prepare(self.ctx, t_write), "kv_paged_prepare")

    def reorder(self, beam_idx: torch.Tensor, t_valid: int):
        _check(lib().kv_paged_reorder(self.ctx, _dev_ptr(beam_idx, "beam_idx", torch.int32), t_valid),
               "kv_paged_reorder")

    def copy(self):
        """Run the copy-on-write tasks that BeamSearch.step_paged recorded."""
        _check(lib().kv_paged_copy(self.ctx), "kv_paged_copy")

    def save(self):
        """Snapshot the allocator state on the device (no host round trip)."""
        _check(lib().kv_paged_save(self.ctx), "kv_paged_save")

    def restore(self):
        """Return the allocator to the last snapshot (no host round trip)."""
        _check(lib().kv_paged_restore(self.ctx), "kv_paged_restore")

    def table(self) -> torch.Tensor:
        """A copy of the block table [R, max_blocks] (int32, on the device)."""
        out = torch.empty(self.R, self.max_blocks, dtype=torch.int32, device=self.device)
        _check(lib().kv_paged_copy_table(self.ctx, _vp(out.data_ptr())), "kv_paged_copy_table")
        return out

    def counts(self):
        """(refcnt [batch * blocks_per_sentence], nblk [R]) as int32 device tensors."""
        rc = torch.empty(self.batch * self.S, dtype=torch.int32, device=self.device)
        nb = torch.empty(self.R, dtype=torch.int32, device=self.device)
        _check(lib().kv_paged_counts(self.ctx, _vp(rc.data_ptr()), _vp(nb.data_ptr())), "kv_paged_counts")
        return rc, nb

    def cow_slots(self) -> int:
        """Filled slots copied by copy-on-write since init (synchronises)."""
        n = _c_i64()
        _check(lib().kv_paged_cow_slots(self.ctx, ctypes.byref(n)), "kv_paged_cow_slots")
        return n.value

    def status(self) -> int:
        return lib().kv_paged_status(self.ctx)

    def close(self):
        if getattr(self, "ctx", None) is not None and self.ctx.value:
            lib().kv_paged_destroy(self.ctx)
            self.ctx = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def bpd_propose(logits: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """Predict: argmax over V of logits [B, k, V] (dense) -> int32 [B, k]."""
    if logits.dim() != 3 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous [B, k, V] tensor")
    B, k, V = logits.shape
    if out is None:
        out = torch.empty(B, k, dtype=torch.int32, device=logits.device)
    _check(lib().bpd_propose(_dev_ptr(logits, "logits"), B, k, V, _dtype_code(logits.dtype),
                             _dev_ptr(out, "out", torch.int32), _stream(logits.device)), "bpd_propose")
    return out


def bpd_verify(logits: torch.Tensor, proposals: torch.Tensor, eos: int = -1, khat: torch.Tensor | None = None,
               next_out: torch.Tensor | None = None, criterion: int = 0, param: int = 0, min_accept: int = 1):
    """Verify + accept on combined logits [B, k, k, V] -> (khat int32 [B], next proposals int32 [B, k]).

    criterion BPD_EXACT (default), BPD_TOPK (param = top-k size) or BPD_DISTANCE (param =
    largest token distance), and min_accept (the minimum accepted block): the relaxed
    verify of bpd_verify_approx."""
    if logits.dim() != 4 or logits.shape[1] != logits.shape[2] or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous [B, k, k, V] tensor")
    B, k, _, V = logits.shape
    if proposals.shape != (B, k) or not proposals.is_contiguous():
        raise ValueError("proposals must be a contiguous [B, k] int32 tensor")
    if khat is None:
        khat = torch.empty(B, dtype=torch.int32, device=logits.device)
    if next_out is None:
        next_out = torch.empty(B, k, dtype=torch.int32, device=logits.device)
    if criterion == BPD_EXACT and min_accept == 1:
        _check(lib().bpd_verify(_dev_ptr(logits, "logits"), _dev_ptr(proposals, "proposals", torch.int32), B, k, V,
                                _dtype_code(logits.dtype), eos, _dev_ptr(khat, "khat", torch.int32),
                                _dev_ptr(next_out, "next", torch.int32), _stream(logits.device)), "bpd_verify")
    else:
        _check(lib().bpd_verify_approx(_dev_ptr(logits, "logits"), _dev_ptr(proposals, "proposals", torch.int32), B,
                                       k, V, _dtype_code(logits.dtype), eos, criterion, param, min_accept,
                                       _dev_ptr(khat, "khat", torch.int32), _dev_ptr(next_out, "next", torch.int32),
                                       _stream(logits.device)), "bpd_verify_approx")
    return khat, next_out


def gather_shard_partials(partial: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather one shard partial per rank (torch.distributed, rank order): [world, bytes].

    Each rank of a vocabulary-parallel LM head holds the columns of one shard; after
    BeamSearch.shard_partial this exchange gives every rank the partials that
    BeamSearch.merge_shards takes.
    """
    import torch.distributed as dist
    world = dist.get_world_size(group)
    out = torch.empty(world, partial.numel(), dtype=partial.dtype, device=partial.device)
    dist.all_gather(list(out.unbind(0)), partial.contiguous(), group=group)
    return out
