"""Engram lookup layer for one GB300 GPU: Python binding of libengram.

Every function here only marshals arguments into the C ABI declared in
``include/engram.h`` (device pointers, sizes, the current CUDA stream) and
allocates output tensors with PyTorch; all computation runs in the CUDA
kernels of ``libengram.so``.  If the library has not been built the first
call raises ``EngramError``; there is no fallback path.

Build: ``python -m hashed_gram_conditional_gb300.build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

__all__ = [
    "EngramError", "Layout", "build_layout", "engram_hash", "engram_hash_all_layers", "engram_hash_step",
    "engram_hash_gather", "engram_hash_gather_step", "engram_hash_gather_fp8", "engram_hash_gather_step_fp8",
    "engram_gather_fp8", "engram_gather_rows_bf16", "engram_hash_gather_rows_bf16", "engram_fill_synthetic_rows_bf16",
    "engram_gather_dequant", "engram_dequant_rows", "engram_host_gather", "engram_host_gather_async",
    "engram_pack_wkv", "engram_project", "engram_gate_add", "engram_fill_synthetic_table",
    "engram_selftest_mod", "engram_project_gate", "project_gate_workspace", "partials_shape", "EngramLayer",
    "library_path", "ST_BAD_TOKEN", "ST_BAD_ROW", "ST_BAD_SLOT", "ST_TIMEOUT", "DEAD", "ROW_BYTES", "DecodeGraph",
    "set_kernel_options", "kernel_options", "sf_cols", "sf_word_index",
]

MAX_LAYERS = 8
MAX_NGRAM = 4
MAX_COLS = 32
DEAD = -1
ROW_BYTES = 264
HEAD_DIM = 256


def sf_cols(n_tokens: int) -> int:
    """Words per k-block row of a block-FP8 scale array for n_tokens positions:
    n_tokens rounded up to a multiple of 128."""
    return (n_tokens + 127) // 128 * 128


def sf_word_index(i):
    """Word of position (or wkv column) i within a k-block row of a block-FP8
    scale array: the 16 bytes at word 4 r of each 128-word block hold rows r,
    r + 32, r + 64 and r + 96 (the image the tensor cores' scale copy reads)."""
    return (i & ~127) | ((i & 31) << 2) | ((i >> 5) & 3)
ST_BAD_TOKEN, ST_BAD_ROW, ST_BAD_SLOT, ST_TIMEOUT = 1, 2, 4, 8

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libengram.so")


def library_path() -> str:
    return _LIB_PATH


class EngramError(RuntimeError):
    pass


class _LayoutParams(ctypes.Structure):
    _fields_ = [
        ("vocab_compressed", ctypes.c_int64),
        ("expected_vocab", ctypes.c_int64),
        ("base_rows", ctypes.c_int64),
        ("n_layers", ctypes.c_int32),
        ("layer_ids", ctypes.c_int32 * MAX_LAYERS),
        ("max_ngram", ctypes.c_int32),
        ("n_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("pad_id", ctypes.c_int32),
        ("use_multiplier_override", ctypes.c_int32),
        ("multiplier_override", (ctypes.c_int64 * MAX_NGRAM) * MAX_LAYERS),
    ]


class _Layout(ctypes.Structure):
    _fields_ = [
        ("vocab_compressed", ctypes.c_int64),
        ("base_rows", ctypes.c_int64),
        ("n_layers", ctypes.c_int32),
        ("max_ngram", ctypes.c_int32),
        ("n_heads", ctypes.c_int32),
        ("n_cols", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("pad_id", ctypes.c_int32),
        ("layer_ids", ctypes.c_int32 * MAX_LAYERS),
        ("total_rows", ctypes.c_int64 * MAX_LAYERS),
        ("primes", (ctypes.c_int64 * MAX_COLS) * MAX_LAYERS),
        ("offsets", (ctypes.c_int64 * MAX_COLS) * MAX_LAYERS),
        ("reciprocal", (ctypes.c_uint64 * MAX_COLS) * MAX_LAYERS),
        ("multipliers", (ctypes.c_int64 * MAX_NGRAM) * MAX_LAYERS),
    ]


_lib = None
_lib_lock = threading.Lock()

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F32 = ctypes.c_float

_SIGS = {
    "engram_build_layout": [ctypes.POINTER(_LayoutParams), ctypes.POINTER(_Layout)],
    "engram_hash": [ctypes.POINTER(_Layout), _I32, _P, _I64, _P, _I32, _P, _I64, _P, _P, _P, _P, _P],
    "engram_hash_step": [ctypes.POINTER(_Layout), _I32, _P, _P, _I32, _P, _I64, _P, _I64, _P, _P, _P, _P],
    "engram_gather_dequant": [_P, _I64, _I64, _P, _I64, _I32, _P, _P, _P],
    "engram_pack_wkv": [_P, _I64, _I64, _P, _P],
    "engram_project": [_P, _I64, _I64, _P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P],
    "engram_gate_add": [_P, _P, _P, _P, _I64, _I32, _I32, _F32, _F32, _F32, _P, _P],
    "engram_fill_synthetic_table": [_P, _I64, ctypes.c_uint64, _P],
    "engram_selftest_mod": [ctypes.POINTER(_Layout), _I32, _P, _I64, _P, _P],
    "engram_project_gate": [_P, _I64, _I64, _P, _I32, _I32, _P, _P, _P, _P, _F32, _F32, _F32, _P, _P,
                            ctypes.c_size_t, _P, _P],
    "engram_hash_all_layers": [ctypes.POINTER(_Layout), _P, _I64, _P, _I32, _P, _I64, _P, _P, _P, _P, _P],
    "engram_dequant_rows": [_P, _I64, _I64, _I32, _P, _P, _P],
    "engram_host_gather": [_P, _I64, _P, _I64, _P, _I32, _P],
    "engram_host_gather_async": [_P, _I64, _P, _I64, _P, _I32, _P, _P],
    "engram_hash_gather": [ctypes.POINTER(_Layout), _I32, _P, _I64, _P, _I32, _P, _I64, _P, _P, _I64, _P, _P, _P, _P,
                           _P],
    "engram_gather_fp8": [_P, _I64, _I64, _P, _I64, _I32, _P, _P, _P, _P],
    "engram_hash_gather_fp8": [ctypes.POINTER(_Layout), _I32, _P, _I64, _P, _I32, _P, _I64, _P, _P, _I64, _P, _P,
                               _P, _P, _P, _P],
    "engram_selftest_wait": [_I32, _P, _P, _P],
    "engram_gather_rows_bf16": [_P, _I64, _I32, _P, _I64, _I32, _P, _P, _P],
    "engram_hash_gather_rows_bf16": [ctypes.POINTER(_Layout), _I32, _P, _I64, _P, _I32, _P, _I64, _P, _P, _I32, _P,
                                     _P, _P, _P, _P],
    "engram_fill_synthetic_rows_bf16": [_P, _I64, _I32, ctypes.c_uint64, _P],
    "engram_hash_gather_step": [ctypes.POINTER(_Layout), _I32, _P, _P, _I32, _P, _I64, _P, _I64, _P, _I64, _P, _P,
                                _P, _P, _P],
    "engram_hash_gather_step_fp8": [ctypes.POINTER(_Layout), _I32, _P, _P, _I32, _P, _I64, _P, _I64, _P, _I64, _P,
                                    _P, _P, _P, _P, _P],
    "engram_pack_wkv_fp8": [_P, _P, _I64, _I64, _P, _P, _P],
    "engram_project_fp8": [_P, _P, _I64, _I64, _P, _P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P],
    "engram_project_gate_fp8": [_P, _P, _I64, _I64, _P, _P, _I32, _I32, _P, _P, _P, _P, _F32, _F32, _F32, _P, _P,
                                ctypes.c_size_t, _P, _P],
    "engram_set_kernel_options": [_P],
    "engram_get_kernel_options": [_P],
    "engram_short_conv_add": [_P, _P, _P, _P, _I64, _I32, _I32, _P, _I64, _P, _P, _P, _I32, _I32, _F32, _P, _P,
                              _I64, _P, ctypes.c_size_t, _P, _P],
}


def _load():
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise EngramError(
                f"CUDA library {_LIB_PATH} is not built; run `python -m hashed_gram_conditional_gb300.build`")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.engram_last_error.restype = ctypes.c_char_p
        lib.engram_status_string.restype = ctypes.c_char_p
        lib.engram_status_string.argtypes = [ctypes.c_int]
        lib.engram_project_partials_bytes.restype = ctypes.c_size_t
        lib.engram_project_partials_bytes.argtypes = [_I64, _I32, _I32]
        lib.engram_project_gate_workspace_bytes.restype = ctypes.c_size_t
        lib.engram_project_gate_workspace_bytes.argtypes = [_I64, _I32, _I32]
        lib.engram_short_conv_workspace_bytes.restype = ctypes.c_size_t
        lib.engram_short_conv_workspace_bytes.argtypes = [_I64, _I32]
        lib.engram_layout_size.restype = ctypes.c_size_t
        lib.engram_layout_params_size.restype = ctypes.c_size_t
        if lib.engram_layout_size() != ctypes.sizeof(_Layout) or \
                lib.engram_layout_params_size() != ctypes.sizeof(_LayoutParams):
            raise EngramError("libengram struct layout does not match the binding")
        _lib = lib
        return lib


def lib():
    """The loaded ctypes library (raises EngramError when it is not built)."""
    return _load()


def _check(rc: int, name: str):
    if rc != 0:
        L = _load()
        raise EngramError(f"{name}: {L.engram_status_string(rc).decode()}: {L.engram_last_error().decode()}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, device=None, numel=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, has {t.numel()}")


class _KernelOptions(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in
                ("projection_cta", "gather_copy", "fp8_pair", "fp8_fused", "plain_launch")]


def kernel_options() -> dict:
    """The engram_kernel_options in force, as a dict (all zero: the library's own choice)."""
    o = _KernelOptions()
    _check(_load().engram_get_kernel_options(ctypes.byref(o)), "engram_get_kernel_options")
    return {name: int(getattr(o, name)) for name, _ in _KernelOptions._fields_}


def set_kernel_options(**opts) -> dict:
    """Override the library's kernel choice process-wide (engram_set_kernel_options).

    Keys: projection_cta (0 default, 1 single CTA, 2 CTA pair), gather_copy
    (0 cp.async, 1 TMA bulk), fp8_pair, fp8_fused, plain_launch (0/1); keys
    not given keep their current value.  Returns the previous options."""
    prev = kernel_options()
    unknown = set(opts) - set(prev)
    if unknown:
        raise ValueError(f"unknown kernel options {sorted(unknown)}")
    o = _KernelOptions(**{**prev, **{k: int(v) for k, v in opts.items()}})
    _check(_load().engram_set_kernel_options(ctypes.byref(o)), "engram_set_kernel_options")
    return prev


# --------------------------------------------------------------------------- layout


class Layout:
    """Immutable table layout (wraps the C struct engram_layout)."""

    def __init__(self, raw: _Layout):
        self._raw = raw

    @property
    def ref(self):
        return ctypes.byref(self._raw)

    @property
    def n_layers(self) -> int:
        return self._raw.n_layers

    @property
    def n_cols(self) -> int:
        return self._raw.n_cols

    @property
    def max_ngram(self) -> int:
        return self._raw.max_ngram

    @property
    def n_heads(self) -> int:
        return self._raw.n_heads

    @property
    def pad_id(self) -> int:
        return self._raw.pad_id

    @property
    def vocab(self) -> int:
        return self._raw.vocab_compressed

    def layer_id(self, layer: int) -> int:
        return self._raw.layer_ids[layer]

    def primes(self, layer: int):
        return [self._raw.primes[layer][j] for j in range(self.n_cols)]

    def offsets(self, layer: int):
        return [self._raw.offsets[layer][j] for j in range(self.n_cols)]

    def total_rows(self, layer: int) -> int:
        return self._raw.total_rows[layer]

    def multipliers(self, layer: int):
        return [self._raw.multipliers[layer][i] for i in range(self.max_ngram)]


def build_layout(vocab: int, base_rows: int, layer_ids: Sequence[int], max_ngram: int = 4, n_heads: int = 8,
                 head_dim: int = 256, pad_id: int = 0, expected_vocab: int = 0,
                 multipliers: Optional[Sequence[Sequence[int]]] = None) -> Layout:
    L = _load()
    p = _LayoutParams()
    p.vocab_compressed = vocab
    p.expected_vocab = expected_vocab
    p.base_rows = base_rows
    if not (1 <= len(layer_ids) <= MAX_LAYERS):
        raise ValueError("1..8 layers")
    p.n_layers = len(layer_ids)
    for i, lid in enumerate(layer_ids):
        p.layer_ids[i] = lid
    p.max_ngram = max_ngram
    p.n_heads = n_heads
    p.head_dim = head_dim
    p.pad_id = pad_id
    if multipliers is not None:
        p.use_multiplier_override = 1
        for i, row in enumerate(multipliers):
            for j, m in enumerate(row):
                p.multiplier_override[i][j] = int(m)
    out = _Layout()
    _check(L.engram_build_layout(ctypes.byref(p), ctypes.byref(out)), "engram_build_layout")
    return Layout(out)


# --------------------------------------------------------------------------- stages


def new_status(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def engram_hash(layout: Layout, layer: int, raw_ids: torch.Tensor, cu_seqlens: torch.Tensor,
                token_map: torch.Tensor, hist: Optional[torch.Tensor] = None,
                row_ids: Optional[torch.Tensor] = None, mask: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None):
    """Prefill hash; returns (row_ids int32 [T][n_cols], mask uint8 [T]). hist is updated in place."""
    L = _load()
    dev = raw_ids.device
    T = raw_ids.numel()
    n_seqs = cu_seqlens.numel() - 1
    _need(raw_ids, "raw_ids", torch.int32)
    _need(cu_seqlens, "cu_seqlens", torch.int64, dev)
    _need(token_map, "token_map", torch.int32, dev)
    if hist is not None:
        _need(hist, "hist", torch.int32, dev, n_seqs * (layout.max_ngram - 1))
    if row_ids is None:
        row_ids = torch.empty((T, layout.n_cols), dtype=torch.int32, device=dev)
    if mask is None:
        mask = torch.empty(T, dtype=torch.uint8, device=dev)
    _need(row_ids, "row_ids", torch.int32, dev, T * layout.n_cols)
    _need(mask, "mask", torch.uint8, dev, T)
    _check(L.engram_hash(layout.ref, layer, _ptr(raw_ids), T, _ptr(cu_seqlens), n_seqs, _ptr(token_map),
                         token_map.numel(), _ptr(hist), _ptr(row_ids), _ptr(mask), _ptr(status), _stream(dev)),
           "engram_hash")
    return row_ids, mask


def engram_hash_all_layers(layout: Layout, raw_ids: torch.Tensor, cu_seqlens: torch.Tensor,
                           token_map: torch.Tensor, hist: Optional[torch.Tensor] = None,
                           row_ids: Optional[torch.Tensor] = None, mask: Optional[torch.Tensor] = None,
                           status: Optional[torch.Tensor] = None):
    """Prefill hash of every layer; returns (row_ids int32 [n_layers][T][n_cols], mask uint8 [T])."""
    L = _load()
    dev = raw_ids.device
    T = raw_ids.numel()
    n_seqs = cu_seqlens.numel() - 1
    _need(raw_ids, "raw_ids", torch.int32)
    _need(cu_seqlens, "cu_seqlens", torch.int64, dev)
    _need(token_map, "token_map", torch.int32, dev)
    if hist is not None:
        _need(hist, "hist", torch.int32, dev, n_seqs * (layout.max_ngram - 1))
    if row_ids is None:
        row_ids = torch.empty((layout.n_layers, T, layout.n_cols), dtype=torch.int32, device=dev)
    if mask is None:
        mask = torch.empty(T, dtype=torch.uint8, device=dev)
    _need(row_ids, "row_ids", torch.int32, dev, layout.n_layers * T * layout.n_cols)
    _need(mask, "mask", torch.uint8, dev, T)
    _check(L.engram_hash_all_layers(layout.ref, _ptr(raw_ids), T, _ptr(cu_seqlens), n_seqs, _ptr(token_map),
                                    token_map.numel(), _ptr(hist), _ptr(row_ids), _ptr(mask), _ptr(status),
                                    _stream(dev)), "engram_hash_all_layers")
    return row_ids, mask


def engram_hash_step(layout: Layout, layer: int, raw_ids: torch.Tensor, slots: torch.Tensor,
                     token_map: torch.Tensor, hist: torch.Tensor, row_ids: Optional[torch.Tensor] = None,
                     mask: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None):
    """One decode step; returns (row_ids [B][n_cols], mask [B]); hist [S][max_ngram-1] updated in place."""
    L = _load()
    dev = raw_ids.device
    B = raw_ids.numel()
    _need(raw_ids, "raw_ids", torch.int32)
    _need(slots, "slots", torch.int32, dev, B)
    _need(token_map, "token_map", torch.int32, dev)
    _need(hist, "hist", torch.int32, dev)
    depth = layout.max_ngram - 1
    if hist.numel() % depth:
        raise ValueError("hist must be [n_slots][max_ngram-1]")
    if row_ids is None:
        row_ids = torch.empty((B, layout.n_cols), dtype=torch.int32, device=dev)
    if mask is None:
        mask = torch.empty(B, dtype=torch.uint8, device=dev)
    _need(row_ids, "row_ids", torch.int32, dev, B * layout.n_cols)
    _need(mask, "mask", torch.uint8, dev, B)
    _check(L.engram_hash_step(layout.ref, layer, _ptr(raw_ids), _ptr(slots), B, _ptr(token_map),
                              token_map.numel(), _ptr(hist), hist.numel() // depth, _ptr(row_ids), _ptr(mask),
                              _ptr(status), _stream(dev)), "engram_hash_step")
    return row_ids, mask


def _step_args(layout: Layout, raw_ids: torch.Tensor, slots: torch.Tensor, token_map: torch.Tensor,
               table: torch.Tensor, hist: torch.Tensor, mask, row_ids):
    """Checks shared by the fused decode steps; returns (B, n_slots, mask)."""
    dev = raw_ids.device
    B = raw_ids.numel()
    _need(raw_ids, "raw_ids", torch.int32)
    _need(slots, "slots", torch.int32, dev, B)
    _need(token_map, "token_map", torch.int32, dev)
    _need(hist, "hist", torch.int32, dev)
    if table.is_cuda:
        _need(table, "table", torch.uint8, dev)
    elif not (table.dtype == torch.uint8 and table.is_pinned() and table.is_contiguous()):
        raise ValueError("a host table must be a contiguous pinned uint8 tensor (read over NVLink-C2C)")
    depth = layout.max_ngram - 1
    if hist.numel() % depth:
        raise ValueError("hist must be [n_slots][max_ngram-1]")
    if mask is None:
        mask = torch.empty(B, dtype=torch.uint8, device=dev)
    _need(mask, "mask", torch.uint8, dev, B)
    if row_ids is not None:
        _need(row_ids, "row_ids", torch.int32, dev, B * layout.n_cols)
    return B, hist.numel() // depth, mask


def engram_hash_gather_step(layout: Layout, layer: int, raw_ids: torch.Tensor, slots: torch.Tensor,
                            token_map: torch.Tensor, table: torch.Tensor, hist: torch.Tensor,
                            e: Optional[torch.Tensor] = None, mask: Optional[torch.Tensor] = None,
                            row_ids: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None):
    """One decode step hashed and gathered in one kernel: returns (e bf16 [B][n_cols*256], mask uint8 [B]);
    hist [S][max_ngram-1] is rolled in place; row_ids is filled only when given."""
    L = _load()
    dev = raw_ids.device
    B, n_slots, mask = _step_args(layout, raw_ids, slots, token_map, table, hist, mask, row_ids)
    C = layout.n_cols
    if e is None:
        e = torch.empty((B, C * HEAD_DIM), dtype=torch.bfloat16, device=dev)
    _need(e, "e", torch.bfloat16, dev, B * C * HEAD_DIM)
    _check(L.engram_hash_gather_step(layout.ref, layer, _ptr(raw_ids), _ptr(slots), B, _ptr(token_map),
                                     token_map.numel(), _ptr(hist), n_slots, _ptr(table), table.numel(), _ptr(e),
                                     _ptr(mask), _ptr(row_ids), _ptr(status), _stream(dev)),
           "engram_hash_gather_step")
    return e, mask


def engram_hash_gather_step_fp8(layout: Layout, layer: int, raw_ids: torch.Tensor, slots: torch.Tensor,
                                token_map: torch.Tensor, table: torch.Tensor, hist: torch.Tensor,
                                e8: Optional[torch.Tensor] = None, sf: Optional[torch.Tensor] = None,
                                mask: Optional[torch.Tensor] = None, row_ids: Optional[torch.Tensor] = None,
                                status: Optional[torch.Tensor] = None):
    """engram_hash_gather_step with FP8 outputs; returns (e8, sf, mask)."""
    L = _load()
    dev = raw_ids.device
    B, n_slots, mask = _step_args(layout, raw_ids, slots, token_map, table, hist, mask, row_ids)
    C = layout.n_cols
    if e8 is None:
        e8 = torch.empty((B, C * HEAD_DIM), dtype=torch.uint8, device=dev)
    if sf is None:
        sf = torch.empty((2 * C, sf_cols(B)), dtype=torch.int32, device=dev)
    _need(e8, "e8", torch.uint8, dev, B * C * HEAD_DIM)
    _need(sf, "sf", torch.int32, dev, 2 * C * sf_cols(B))
    _check(L.engram_hash_gather_step_fp8(layout.ref, layer, _ptr(raw_ids), _ptr(slots), B, _ptr(token_map),
                                         token_map.numel(), _ptr(hist), n_slots, _ptr(table), table.numel(),
                                         _ptr(e8), _ptr(sf), _ptr(mask), _ptr(row_ids), _ptr(status), _stream(dev)),
           "engram_hash_gather_step_fp8")
    return e8, sf, mask


def engram_gather_dequant(table: torch.Tensor, total_rows: int, row_ids: torch.Tensor,
                          e: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Gather and dequantise: returns e bf16 [T][n_cols*256]."""
    L = _load()
    dev = row_ids.device
    if table.is_cuda:
        _need(table, "table", torch.uint8, dev)
    elif not (table.dtype == torch.uint8 and table.is_pinned() and table.is_contiguous()):
        raise ValueError("a host table must be a contiguous pinned uint8 tensor (read over NVLink-C2C)")
    _need(row_ids, "row_ids", torch.int32)
    T, C = row_ids.shape
    if e is None:
        e = torch.empty((T, C * HEAD_DIM), dtype=torch.bfloat16, device=dev)
    _need(e, "e", torch.bfloat16, dev, T * C * HEAD_DIM)
    _check(L.engram_gather_dequant(_ptr(table), total_rows, table.numel(), _ptr(row_ids), T, C, _ptr(e),
                                   _ptr(status), _stream(dev)), "engram_gather_dequant")
    return e


def engram_hash_gather(layout: Layout, layer: int, raw_ids: torch.Tensor, cu_seqlens: torch.Tensor,
                       token_map: torch.Tensor, table: torch.Tensor, hist: Optional[torch.Tensor] = None,
                       e: Optional[torch.Tensor] = None, mask: Optional[torch.Tensor] = None,
                       row_ids: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None):
    """Hash + gather + dequantise in one kernel; returns (e bf16 [T][n_cols*256], mask uint8 [T]).
    row_ids (int32 [T][n_cols]) is filled only when given; hist is advanced in place."""
    L = _load()
    dev = raw_ids.device
    T = raw_ids.numel()
    C = layout.n_cols
    _need(raw_ids, "raw_ids", torch.int32)
    _need(cu_seqlens, "cu_seqlens", torch.int64, dev)
    _need(token_map, "token_map", torch.int32, dev)
    if table.is_cuda:
        _need(table, "table", torch.uint8, dev)
    elif not (table.dtype == torch.uint8 and table.is_pinned() and table.is_contiguous()):
        raise ValueError("a host table must be a contiguous pinned uint8 tensor (read over NVLink-C2C)")
    n_seqs = cu_seqlens.numel() - 1
    if hist is not None:
        _need(hist, "hist", torch.int32, dev, n_seqs * (layout.max_ngram - 1))
    if e is None:
        e = torch.empty((T, C * HEAD_DIM), dtype=torch.bfloat16, device=dev)
    if mask is None:
        mask = torch.empty(T, dtype=torch.uint8, device=dev)
    _need(e, "e", torch.bfloat16, dev, T * C * HEAD_DIM)
    _need(mask, "mask", torch.uint8, dev, T)
    if row_ids is not None:
        _need(row_ids, "row_ids", torch.int32, dev, T * C)
    _check(L.engram_hash_gather(layout.ref, layer, _ptr(raw_ids), T, _ptr(cu_seqlens), n_seqs, _ptr(token_map),
                                token_map.numel(), _ptr(hist), _ptr(table), table.numel(), _ptr(e), _ptr(mask),
                                _ptr(row_ids), _ptr(status), _stream(dev)), "engram_hash_gather")
    return e, mask


def engram_gather_fp8(table: torch.Tensor, total_rows: int, row_ids: torch.Tensor,
                      e8: Optional[torch.Tensor] = None, sf: Optional[torch.Tensor] = None,
                      status: Optional[torch.Tensor] = None):
    """Gather without dequantising: (e8 uint8 [T][n_cols*256], sf int32 [n_cols*2][sf_cols(T)] words of 4 E8M0
    scales, positions in sf_word_index order)."""
    L = _load()
    dev = row_ids.device
    _need(table, "table", torch.uint8, dev)
    _need(row_ids, "row_ids", torch.int32)
    T, C = row_ids.shape
    if e8 is None:
        e8 = torch.empty((T, C * HEAD_DIM), dtype=torch.uint8, device=dev)
    if sf is None:
        sf = torch.empty((2 * C, sf_cols(T)), dtype=torch.int32, device=dev)
    _need(e8, "e8", torch.uint8, dev, T * C * HEAD_DIM)
    _need(sf, "sf", torch.int32, dev, 2 * C * sf_cols(T))
    _check(L.engram_gather_fp8(_ptr(table), total_rows, table.numel(), _ptr(row_ids), T, C, _ptr(e8), _ptr(sf),
                               _ptr(status), _stream(dev)), "engram_gather_fp8")
    return e8, sf


def engram_hash_gather_fp8(layout: Layout, layer: int, raw_ids: torch.Tensor, cu_seqlens: torch.Tensor,
                           token_map: torch.Tensor, table: torch.Tensor, hist: Optional[torch.Tensor] = None,
                           e8: Optional[torch.Tensor] = None, sf: Optional[torch.Tensor] = None,
                           mask: Optional[torch.Tensor] = None, row_ids: Optional[torch.Tensor] = None,
                           status: Optional[torch.Tensor] = None):
    """Hash + gather, FP8 outputs; returns (e8, sf, mask)."""
    L = _load()
    dev = raw_ids.device
    T = raw_ids.numel()
    C = layout.n_cols
    _need(raw_ids, "raw_ids", torch.int32)
    _need(cu_seqlens, "cu_seqlens", torch.int64, dev)
    _need(token_map, "token_map", torch.int32, dev)
    _need(table, "table", torch.uint8, dev)
    n_seqs = cu_seqlens.numel() - 1
    if hist is not None:
        _need(hist, "hist", torch.int32, dev, n_seqs * (layout.max_ngram - 1))
    if e8 is None:
        e8 = torch.empty((T, C * HEAD_DIM), dtype=torch.uint8, device=dev)
    if sf is None:
        sf = torch.empty((2 * C, sf_cols(T)), dtype=torch.int32, device=dev)
    if mask is None:
        mask = torch.empty(T, dtype=torch.uint8, device=dev)
    _need(e8, "e8", torch.uint8, dev, T * C * HEAD_DIM)
    _need(sf, "sf", torch.int32, dev, 2 * C * sf_cols(T))
    _need(mask, "mask", torch.uint8, dev, T)
    if row_ids is not None:
        _need(row_ids, "row_ids", torch.int32, dev, T * C)
    _check(L.engram_hash_gather_fp8(layout.ref, layer, _ptr(raw_ids), T, _ptr(cu_seqlens), n_seqs, _ptr(token_map),
                                    token_map.numel(), _ptr(hist), _ptr(table), table.numel(), _ptr(e8), _ptr(sf),
                                    _ptr(mask), _ptr(row_ids), _ptr(status), _stream(dev)), "engram_hash_gather_fp8")
    return e8, sf, mask


def engram_pack_wkv_fp8(w8: torch.Tensor, sf: torch.Tensor):
    """Block-FP8 wkv (codes uint8 [K][N], scales uint8 [K/32][N]) -> (packed codes, packed scale words
    [K/128][N], the columns of each 128 in sf_word_index order)."""
    L = _load()
    dev = w8.device
    K, N = w8.shape
    _need(w8, "w8", torch.uint8, dev)
    _need(sf, "sf", torch.uint8, dev, (K // 32) * N)
    w8p = torch.empty(K * N, dtype=torch.uint8, device=dev)
    sfp = torch.empty((K // 128, N), dtype=torch.int32, device=dev)
    _check(L.engram_pack_wkv_fp8(_ptr(w8), _ptr(sf), K, N, _ptr(w8p), _ptr(sfp), _stream(dev)),
           "engram_pack_wkv_fp8")
    return w8p, sfp


def engram_project_fp8(e8: torch.Tensor, sfa: torch.Tensor, w8p: torch.Tensor, sfb: torch.Tensor, h: torch.Tensor,
                       q_w: torch.Tensor, k_w: torch.Tensor, partials: Optional[torch.Tensor] = None,
                       v: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None):
    """engram_project on FP8 operands; returns (partials, v)."""
    L = _load()
    dev = e8.device
    _need(e8, "e8", torch.uint8)
    T, K = e8.shape
    _need(h, "h", torch.bfloat16, dev)
    _, hc, H = h.shape
    _need(sfa, "sfa", torch.int32, dev, (K // 128) * sf_cols(T))
    _need(w8p, "w8p", torch.uint8, dev, K * (hc + 1) * H)
    _need(sfb, "sfb", torch.int32, dev, (K // 128) * (hc + 1) * H)
    if partials is None:
        partials = torch.empty(partials_shape(T, H, hc), dtype=torch.float32, device=dev)
    if v is None:
        v = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    _need(partials, "partials", torch.float32, dev, T * hc * (H // 256) * 4)
    _need(v, "v", torch.bfloat16, dev, T * H)
    _check(L.engram_project_fp8(_ptr(e8), _ptr(sfa), T, K, _ptr(w8p), _ptr(sfb), H, hc, _ptr(h), _ptr(q_w), _ptr(k_w),
                                _ptr(partials), _ptr(v), _ptr(status), _stream(dev)), "engram_project_fp8")
    return partials, v


def engram_project_gate_fp8(e8: torch.Tensor, sfa: torch.Tensor, w8p: torch.Tensor, sfb: torch.Tensor,
                            h: torch.Tensor, q_w: torch.Tensor, k_w: torch.Tensor, mask: Optional[torch.Tensor],
                            eps: float = 1e-6, clamp: float = 1e-6, score_scale: Optional[float] = None,
                            gate_out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                            status: Optional[torch.Tensor] = None):
    """engram_project_gate on FP8 operands: h updated in place; returns gate_out (or None)."""
    L = _load()
    dev = e8.device
    _need(e8, "e8", torch.uint8)
    T, K = e8.shape
    _need(h, "h", torch.bfloat16, dev)
    _, hc, H = h.shape
    _need(sfa, "sfa", torch.int32, dev, (K // 128) * sf_cols(T))
    _need(w8p, "w8p", torch.uint8, dev, K * (hc + 1) * H)
    _need(sfb, "sfb", torch.int32, dev, (K // 128) * (hc + 1) * H)
    if mask is not None:
        _need(mask, "mask", torch.uint8, dev, T)
    if gate_out is not None:
        _need(gate_out, "gate_out", torch.float32, dev, T * hc)
    if workspace is None:
        workspace = project_gate_workspace(T, H, hc, dev)
    if score_scale is None:
        score_scale = H ** -0.5
    _check(L.engram_project_gate_fp8(_ptr(e8), _ptr(sfa), T, K, _ptr(w8p), _ptr(sfb), H, hc, _ptr(h), _ptr(q_w),
                                     _ptr(k_w), _ptr(mask), eps, clamp, score_scale, _ptr(gate_out), _ptr(workspace),
                                     workspace.numel(), _ptr(status), _stream(dev)), "engram_project_gate_fp8")
    return gate_out


def engram_dequant_rows(rows: torch.Tensor, n_cols: int, e: Optional[torch.Tensor] = None,
                        status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Dequantise contiguous device rows uint8 [n][264] -> e bf16 [n/n_cols][n_cols*256]."""
    L = _load()
    dev = rows.device
    _need(rows, "rows", torch.uint8)
    n = rows.numel() // ROW_BYTES
    if e is None:
        e = torch.empty((n // n_cols, n_cols * HEAD_DIM), dtype=torch.bfloat16, device=dev)
    _need(e, "e", torch.bfloat16, dev, n * HEAD_DIM)
    _check(L.engram_dequant_rows(_ptr(rows), n, rows.numel(), n_cols, _ptr(e), _ptr(status), _stream(dev)),
           "engram_dequant_rows")
    return e


def _host_ptr(a):
    """Address of a host buffer: a CPU torch tensor or a numpy array (contiguous)."""
    if isinstance(a, torch.Tensor):
        if a.is_cuda or not a.is_contiguous():
            raise ValueError("host buffers must be contiguous CPU tensors")
        return ctypes.c_void_p(a.data_ptr())
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("host buffers must be C-contiguous")
    return ctypes.c_void_p(a.ctypes.data)


def engram_host_gather(table, total_rows: int, row_ids, staging, n_threads: int = 0) -> int:
    """Copy table rows row_ids (host) into staging (host); returns the count of out-of-range ids."""
    L = _load()
    n = (row_ids.numel() if isinstance(row_ids, torch.Tensor) else row_ids.size)
    nbytes = staging.numel() if isinstance(staging, torch.Tensor) else staging.nbytes
    if nbytes < n * ROW_BYTES:
        raise ValueError("staging buffer too small")
    bad = ctypes.c_int64(0)
    _check(L.engram_host_gather(_host_ptr(table), total_rows, _host_ptr(row_ids), n, _host_ptr(staging), n_threads,
                                ctypes.byref(bad)), "engram_host_gather")
    return bad.value


def engram_host_gather_async(table: torch.Tensor, total_rows: int, row_ids: torch.Tensor, staging: torch.Tensor,
                             bad_rows: torch.Tensor, stream: torch.cuda.Stream, n_threads: int = 0):
    """Enqueue the host gather on `stream` (after work already on it); bad_rows: int64 CPU tensor [1]."""
    L = _load()
    if bad_rows.dtype != torch.int64 or bad_rows.is_cuda:
        raise TypeError("bad_rows must be a CPU int64 tensor")
    n = row_ids.numel()
    if staging.numel() < n * ROW_BYTES:
        raise ValueError("staging buffer too small")
    _check(L.engram_host_gather_async(_host_ptr(table), total_rows, _host_ptr(row_ids), n, _host_ptr(staging),
                                      n_threads, ctypes.c_void_p(bad_rows.data_ptr()),
                                      ctypes.c_void_p(stream.cuda_stream)), "engram_host_gather_async")


def engram_pack_wkv(wkv: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """[K][N] bf16 -> K-major [N][K] bf16 operand layout."""
    L = _load()
    _need(wkv, "wkv", torch.bfloat16)
    K, N = wkv.shape
    if out is None:
        out = torch.empty((N, K), dtype=torch.bfloat16, device=wkv.device)
    _need(out, "out", torch.bfloat16, wkv.device, N * K)
    _check(L.engram_pack_wkv(_ptr(wkv), K, N, _ptr(out), _stream(wkv.device)), "engram_pack_wkv")
    return out


def partials_shape(n_tokens: int, hidden: int, hc: int):
    return (n_tokens, hc, hidden // 256, 4)


def engram_project(e: torch.Tensor, wkv_packed: torch.Tensor, h: torch.Tensor, q_w: torch.Tensor,
                   k_w: torch.Tensor, partials: Optional[torch.Tensor] = None, v: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None):
    """Tensor-core projection; returns (partials f32 [T][hc][H/256][4], v bf16 [T][H])."""
    L = _load()
    dev = e.device
    _need(e, "e", torch.bfloat16)
    T, K = e.shape
    _need(h, "h", torch.bfloat16, dev)
    if h.dim() != 3 or h.shape[0] != T:
        raise ValueError("h must be [T][hc][H]")
    hc, H = h.shape[1], h.shape[2]
    _need(wkv_packed, "wkv_packed", torch.bfloat16, dev, (hc + 1) * H * K)
    _need(q_w, "q_w", torch.float32, dev, H * hc)
    _need(k_w, "k_w", torch.float32, dev, H * hc)
    if partials is None:
        partials = torch.empty(partials_shape(T, H, hc), dtype=torch.float32, device=dev)
    if v is None:
        v = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    _need(partials, "partials", torch.float32, dev, T * hc * (H // 256) * 4)
    _need(v, "v", torch.bfloat16, dev, T * H)
    _check(L.engram_project(_ptr(e), T, K, _ptr(wkv_packed), H, hc, _ptr(h), _ptr(q_w), _ptr(k_w),
                            _ptr(partials), _ptr(v), _ptr(status), _stream(dev)), "engram_project")
    return partials, v


def engram_gate_add(partials: torch.Tensor, v: torch.Tensor, h: torch.Tensor, mask: Optional[torch.Tensor],
                    eps: float = 1e-6, clamp: float = 1e-6, score_scale: Optional[float] = None,
                    gate_out: Optional[torch.Tensor] = None) -> Optional[torch.Tensor]:
    """h <- bf16(h + gate * v) in place; returns gate_out (f32 [T][hc]) when given."""
    L = _load()
    dev = h.device
    _need(h, "h", torch.bfloat16)
    T, hc, H = h.shape
    _need(partials, "partials", torch.float32, dev, T * hc * (H // 256) * 4)
    _need(v, "v", torch.bfloat16, dev, T * H)
    if mask is not None:
        _need(mask, "mask", torch.uint8, dev, T)
    if gate_out is not None:
        _need(gate_out, "gate_out", torch.float32, dev, T * hc)
    if score_scale is None:
        score_scale = H ** -0.5
    _check(L.engram_gate_add(_ptr(partials), _ptr(v), _ptr(h), _ptr(mask), T, H, hc, eps, clamp, score_scale,
                             _ptr(gate_out), _stream(dev)), "engram_gate_add")
    return gate_out


def engram_gates(partials: torch.Tensor, n_tokens: int, hidden: int, hc: int, mask: Optional[torch.Tensor],
                 eps: float = 1e-6, clamp: float = 1e-6, score_scale: Optional[float] = None,
                 gate_out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The gates alone (engram_gate_add without h): f32 [T][hc]."""
    L = _load()
    dev = partials.device
    T = n_tokens
    _need(partials, "partials", torch.float32, dev, T * hc * (hidden // 256) * 4)
    if mask is not None:
        _need(mask, "mask", torch.uint8, dev, T)
    if gate_out is None:
        gate_out = torch.empty((T, hc), dtype=torch.float32, device=dev)
    _need(gate_out, "gate_out", torch.float32, dev, T * hc)
    if score_scale is None:
        score_scale = hidden ** -0.5
    _check(L.engram_gate_add(_ptr(partials), None, None, _ptr(mask), T, hidden, hc, eps, clamp, score_scale,
                             _ptr(gate_out), _stream(dev)), "engram_gate_add")
    return gate_out


def short_conv_workspace(n_tokens: int, hc: int, device) -> torch.Tensor:
    n = _load().engram_short_conv_workspace_bytes(n_tokens, hc)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device)


def engram_short_conv_add(gate: torch.Tensor, v: torch.Tensor, h: torch.Tensor, mask: Optional[torch.Tensor],
                          conv_w: torch.Tensor, gamma: torch.Tensor, dilation: int, eps: float = 1e-6,
                          cu_seqlens: Optional[torch.Tensor] = None, slots: Optional[torch.Tensor] = None,
                          state: Optional[torch.Tensor] = None, state_head: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None):
    """h <- bf16(h + g*bf16(v) + SiLU(conv(RMSNorm(g*bf16(v))))) in place.

    gate f32 [T][hc]; v bf16 [T][H]; h bf16 [T][hc][H]; conv_w f32 [K][hc][H];
    gamma f32 [hc][H]; cu_seqlens int64 [S+1] (None: each position is its own
    sequence); slots int32 [S]; state f32 [n_slots][(K-1)*dilation][hc][H] with
    state_head int32 [n_slots], or None.
    """
    L = _load()
    dev = h.device
    _need(h, "h", torch.bfloat16)
    T, hc, H = h.shape
    _need(gate, "gate", torch.float32, dev, T * hc)
    _need(v, "v", torch.bfloat16, dev, T * H)
    if mask is not None:
        _need(mask, "mask", torch.uint8, dev, T)
    K = conv_w.shape[0]
    _need(conv_w, "conv_w", torch.float32, dev, K * hc * H)
    _need(gamma, "gamma", torch.float32, dev, hc * H)
    n_seqs = T
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int64, dev)
        n_seqs = cu_seqlens.numel() - 1
    if slots is not None:
        _need(slots, "slots", torch.int32, dev, n_seqs)
    n_slots = 0
    if state is not None:
        n_slots = state.shape[0]
        _need(state, "state", torch.float32, dev, n_slots * max((K - 1) * dilation, 1) * hc * H)
        _need(state_head, "state_head", torch.int32, dev, n_slots)
    if workspace is None:
        workspace = short_conv_workspace(T, hc, dev)
    _check(L.engram_short_conv_add(_ptr(gate), _ptr(v), _ptr(h), _ptr(mask), T, H, hc, _ptr(cu_seqlens), n_seqs,
                                   _ptr(slots), _ptr(conv_w), _ptr(gamma), K, dilation, eps, _ptr(state),
                                   _ptr(state_head), n_slots, _ptr(workspace), workspace.numel(), _ptr(status),
                                   _stream(dev)), "engram_short_conv_add")
    return h


def project_gate_workspace(n_tokens: int, hidden: int, hc: int, device) -> torch.Tensor:
    """Workspace tensor for engram_project_gate (torch allocations are 256-byte aligned)."""
    n = _load().engram_project_gate_workspace_bytes(n_tokens, hidden, hc)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device)


def engram_project_gate(e: torch.Tensor, wkv_packed: torch.Tensor, h: torch.Tensor, q_w: torch.Tensor,
                        k_w: torch.Tensor, mask: Optional[torch.Tensor], eps: float = 1e-6, clamp: float = 1e-6,
                        score_scale: Optional[float] = None, gate_out: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None):
    """Fused projection + gate + residual: h <- bf16(h + g * bf16(v)) in place; returns gate_out."""
    L = _load()
    dev = e.device
    _need(e, "e", torch.bfloat16)
    T, K = e.shape
    _need(h, "h", torch.bfloat16, dev)
    if h.dim() != 3 or h.shape[0] != T:
        raise ValueError("h must be [T][hc][H]")
    hc, H = h.shape[1], h.shape[2]
    _need(wkv_packed, "wkv_packed", torch.bfloat16, dev, (hc + 1) * H * K)
    _need(q_w, "q_w", torch.float32, dev, H * hc)
    _need(k_w, "k_w", torch.float32, dev, H * hc)
    if mask is not None:
        _need(mask, "mask", torch.uint8, dev, T)
    if gate_out is not None:
        _need(gate_out, "gate_out", torch.float32, dev, T * hc)
    if workspace is None:
        workspace = project_gate_workspace(T, H, hc, dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if score_scale is None:
        score_scale = H ** -0.5
    _check(L.engram_project_gate(_ptr(e), T, K, _ptr(wkv_packed), H, hc, _ptr(h), _ptr(q_w), _ptr(k_w), _ptr(mask),
                                 eps, clamp, score_scale, _ptr(gate_out), _ptr(workspace), workspace.numel(),
                                 _ptr(status), _stream(dev)), "engram_project_gate")
    return gate_out


def engram_gather_rows_bf16(table: torch.Tensor, row_ids: torch.Tensor, e: Optional[torch.Tensor] = None,
                            status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Gather from a table of plain bf16 rows (bf16 [total_rows][row_dim]):
    returns e bf16 [T][n_cols*row_dim], the rows concatenated as stored."""
    L = _load()
    dev = row_ids.device
    _need(table, "table", torch.bfloat16, dev)
    if table.dim() != 2:
        raise ValueError("a bf16-row table is [total_rows][row_dim]")
    _need(row_ids, "row_ids", torch.int32, dev)
    T, C = row_ids.shape
    R = table.shape[1]
    if e is None:
        e = torch.empty((T, C * R), dtype=torch.bfloat16, device=dev)
    _need(e, "e", torch.bfloat16, dev, T * C * R)
    _check(L.engram_gather_rows_bf16(_ptr(table), table.shape[0], R, _ptr(row_ids), T, C, _ptr(e), _ptr(status),
                                     _stream(dev)), "engram_gather_rows_bf16")
    return e


def engram_hash_gather_rows_bf16(layout: Layout, layer: int, raw_ids: torch.Tensor, cu_seqlens: torch.Tensor,
                                 token_map: torch.Tensor, table: torch.Tensor, hist: Optional[torch.Tensor] = None,
                                 e: Optional[torch.Tensor] = None, mask: Optional[torch.Tensor] = None,
                                 row_ids: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None):
    """Hash + gather from a bf16-row table in one kernel, then the history commit;
    returns (e bf16 [T][n_cols*row_dim], mask uint8 [T])."""
    L = _load()
    dev = raw_ids.device
    T = raw_ids.numel()
    C = layout.n_cols
    _need(raw_ids, "raw_ids", torch.int32)
    _need(cu_seqlens, "cu_seqlens", torch.int64, dev)
    _need(token_map, "token_map", torch.int32, dev)
    _need(table, "table", torch.bfloat16, dev)
    if table.dim() != 2 or table.shape[0] < layout.total_rows(layer):
        raise ValueError("the bf16-row table must be [>= total_rows][row_dim]")
    R = table.shape[1]
    n_seqs = cu_seqlens.numel() - 1
    if hist is not None:
        _need(hist, "hist", torch.int32, dev, n_seqs * (layout.max_ngram - 1))
    if e is None:
        e = torch.empty((T, C * R), dtype=torch.bfloat16, device=dev)
    if mask is None:
        mask = torch.empty(T, dtype=torch.uint8, device=dev)
    _need(e, "e", torch.bfloat16, dev, T * C * R)
    _need(mask, "mask", torch.uint8, dev, T)
    if row_ids is not None:
        _need(row_ids, "row_ids", torch.int32, dev, T * C)
    _check(L.engram_hash_gather_rows_bf16(layout.ref, layer, _ptr(raw_ids), T, _ptr(cu_seqlens), n_seqs,
                                          _ptr(token_map), token_map.numel(), _ptr(hist), _ptr(table), R, _ptr(e),
                                          _ptr(mask), _ptr(row_ids), _ptr(status), _stream(dev)),
           "engram_hash_gather_rows_bf16")
    return e, mask


def engram_fill_synthetic_rows_bf16(table: torch.Tensor, seed: int) -> torch.Tensor:
    """Fill a device bf16-row table [n_rows][row_dim] with the seeded synthetic rows."""
    L = _load()
    _need(table, "table", torch.bfloat16)
    if table.dim() != 2:
        raise ValueError("a bf16-row table is [n_rows][row_dim]")
    _check(L.engram_fill_synthetic_rows_bf16(_ptr(table), table.shape[0], table.shape[1], seed,
                                             _stream(table.device)), "engram_fill_synthetic_rows_bf16")
    return table


def engram_fill_synthetic_table(table: torch.Tensor, n_rows: int, seed: int,
                                device: Optional[torch.device] = None) -> torch.Tensor:
    """Fill a device table, or a pinned host table (written by the kernel through
    its mapped address), with the seeded synthetic rows."""
    L = _load()
    if table.is_cuda:
        _need(table, "table", torch.uint8)
        device = table.device
    elif not (table.dtype == torch.uint8 and table.is_pinned() and table.is_contiguous()):
        raise ValueError("a host table must be a contiguous pinned uint8 tensor")
    elif device is None:
        device = torch.device("cuda", torch.cuda.current_device())
    if table.numel() < n_rows * ROW_BYTES:
        raise ValueError("table too small")
    _check(L.engram_fill_synthetic_table(_ptr(table), n_rows, seed, _stream(device)),
           "engram_fill_synthetic_table")
    return table


def engram_selftest_mod(layout: Layout, layer: int, x: torch.Tensor) -> torch.Tensor:
    """x: uint64 values stored in an int64 tensor; returns int64 [n][n_cols]."""
    L = _load()
    _need(x, "x", torch.int64)
    out = torch.empty((x.numel(), layout.n_cols), dtype=torch.int64, device=x.device)
    _check(L.engram_selftest_mod(layout.ref, layer, _ptr(x), x.numel(), _ptr(out), _stream(x.device)),
           "engram_selftest_mod")
    return out


# --------------------------------------------------------------------------- layer


def engram_selftest_wait(which: int, status: torch.Tensor, scratch: Optional[torch.Tensor] = None):
    """Diagnostic: a bounded wait that nothing satisfies (which 0: an mbarrier
    phase, 1: a global counter) runs out after about a second and sets
    ST_TIMEOUT in ``status``; asynchronous on the current stream."""
    L = _load()
    dev = status.device
    _need(status, "status", torch.int32, dev, 1)
    if scratch is None:
        scratch = torch.empty(2, dtype=torch.int32, device=dev)
    _need(scratch, "scratch", torch.int32, dev, 2)
    _check(L.engram_selftest_wait(which, _ptr(scratch), _ptr(status), _stream(dev)), "engram_selftest_wait")
    return scratch


class EngramLayer:
    """One Engram layer with resident weights: table, token map, packed wkv, q_w, k_w.

    ``prefill`` runs hash -> gather -> fused project/gate on the current
    stream and updates the residual ``h`` in place (``fused=False`` runs the
    projection and the gate kernel separately).

    ``wkv_packed`` is either the bf16 wkv from ``engram_pack_wkv`` or the pair
    (w8p, sfb) from ``engram_pack_wkv_fp8`` (block-FP8 weights): the layer then
    gathers the rows as stored (E4M3 + E8M0) and runs the block-scaled FP8
    projection ([P-O1] §2.3).

    The table may be a device tensor or a pinned host tensor (Grace memory).
    ``prefetch`` + ``prefill_prefetched`` split the layer at the point the
    Engram pages use for offloading: the rows a batch needs depend only on its
    token ids, so they can be fetched while earlier work runs, and the layer
    later only waits for them.
    """

    def __init__(self, layout: Layout, layer: int, table: torch.Tensor, token_map: torch.Tensor,
                 wkv_packed: torch.Tensor, q_w: torch.Tensor, k_w: torch.Tensor, eps: float = 1e-6,
                 clamp: float = 1e-6, score_scale: Optional[float] = None, fused: bool = True,
                 conv: Optional["ShortConv"] = None):
        self.conv = conv
        self.layout, self.layer = layout, layer
        self.table, self.token_map = table, token_map
        self.fp8 = isinstance(wkv_packed, (tuple, list))
        if self.fp8:
            self.w8p, self.sfb = wkv_packed
            if table.dtype != torch.uint8:
                raise ValueError("block-FP8 weights go with the E4M3 + E8M0 row table")
        self.wkv_packed, self.q_w, self.k_w = wkv_packed, q_w, k_w
        self.hidden, self.hc = q_w.shape[0], q_w.shape[1]
        self.eps, self.clamp = eps, clamp
        self.score_scale = self.hidden ** -0.5 if score_scale is None else score_scale
        self.total_rows = layout.total_rows(layer)
        # a bf16 [rows][row_dim] table holds plain rows (generic shapes); a uint8
        # table holds the 264-byte E4M3 + E8M0 rows
        self.row_dim = table.shape[1] if table.dtype == torch.bfloat16 else None
        self.e_dim = layout.n_cols * (self.row_dim if self.row_dim is not None else HEAD_DIM)
        self.fused = fused
        self._ws = {}
        self._pf = {}          # T -> [two prefetch slots]
        self._pf_next = 0

    def _buffers(self, T: int, device):
        key = (T, str(device))
        if key not in self._ws:
            self._ws = {key: dict(
                rows=torch.empty((T, self.layout.n_cols), dtype=torch.int32, device=device),
                mask=torch.empty(T, dtype=torch.uint8, device=device),
                e=torch.empty((T, self.e_dim), dtype=torch.bfloat16, device=device) if not self.fp8 else None,
                e8=torch.empty((T, self.e_dim), dtype=torch.uint8, device=device) if self.fp8 else None,
                sf=torch.empty((2 * self.layout.n_cols, sf_cols(T)), dtype=torch.int32, device=device)
                if self.fp8 else None,
                partials=torch.empty(partials_shape(T, self.hidden, self.hc), dtype=torch.float32, device=device),
                v=torch.empty((T, self.hidden), dtype=torch.bfloat16, device=device),
                work=project_gate_workspace(T, self.hidden, self.hc, device),
                gate=torch.empty((T, self.hc), dtype=torch.float32, device=device),
                conv_ws=short_conv_workspace(T, self.hc, device),
            )}
        return self._ws[key]

    def new_conv_state(self, n_slots: int, device) -> tuple:
        """A zeroed short-convolution state (ring, head) for n_slots sequences."""
        c = self.conv
        R = (c.w.shape[0] - 1) * c.dilation
        return (torch.zeros((n_slots, max(R, 1), self.hc, self.hidden), dtype=torch.float32, device=device),
                torch.zeros(n_slots, dtype=torch.int32, device=device))

    def prefill(self, raw_ids: torch.Tensor, cu_seqlens: torch.Tensor, h: torch.Tensor,
                hist: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                gate_out: Optional[torch.Tensor] = None, conv_state: Optional[tuple] = None):
        """conv_state: (ring, head) from new_conv_state, one slot per sequence, for a
        layer with the short convolution (None: zeros before every sequence)."""
        T = raw_ids.numel()
        b = self._buffers(T, raw_ids.device)
        if self.row_dim is not None:
            engram_hash_gather_rows_bf16(self.layout, self.layer, raw_ids, cu_seqlens, self.token_map, self.table,
                                         hist, b["e"], b["mask"], b["rows"], status)
        elif self.fp8:
            engram_hash_gather_fp8(self.layout, self.layer, raw_ids, cu_seqlens, self.token_map, self.table, hist,
                                   b["e8"], b["sf"], b["mask"], b["rows"], status)
        else:
            engram_hash_gather(self.layout, self.layer, raw_ids, cu_seqlens, self.token_map, self.table, hist,
                               b["e"], b["mask"], b["rows"], status)
        self._gate(b, h, status, gate_out, cu_seqlens=cu_seqlens, conv_state=conv_state)
        return b

    def _prefetch_slot(self, T: int, device):
        key = (T, str(device))
        if key not in self._pf:
            C = self.layout.n_cols
            host = not self.table.is_cuda
            fp8 = self.fp8
            self._pf = {key: [dict(
                rows=torch.empty((T, C), dtype=torch.int32, device=device),
                mask=torch.empty(T, dtype=torch.uint8, device=device),
                e=torch.empty((T, C * HEAD_DIM), dtype=torch.bfloat16, device=device) if not fp8 else None,
                e8=torch.empty((T, C * HEAD_DIM), dtype=torch.uint8, device=device) if fp8 else None,
                sf=torch.empty((2 * C, sf_cols(T)), dtype=torch.int32, device=device) if fp8 else None,
                # the staged rows in order: row t*C + j of the staging buffer is column j of position t
                staged_ids=(torch.arange(T * C, dtype=torch.int32, device=device).view(T, C)
                            if fp8 and host else None),
                rows_h=torch.empty((T, C), dtype=torch.int32, pin_memory=True) if host else None,
                staging=torch.empty(T * C * ROW_BYTES, dtype=torch.uint8, pin_memory=True) if host else None,
                staged=torch.empty(T * C * ROW_BYTES, dtype=torch.uint8, device=device) if host else None,
                bad=torch.zeros(1, dtype=torch.int64),
                consumed=torch.cuda.Event(), busy=False) for _ in range(2)]}
        slot = self._pf[key][self._pf_next]
        if slot["busy"]:
            raise EngramError("two prefetched batches are already waiting; run prefill_prefetched first")
        self._pf_next ^= 1
        return slot

    def prefetch(self, raw_ids: torch.Tensor, cu_seqlens: torch.Tensor, hist: Optional[torch.Tensor] = None,
                 status: Optional[torch.Tensor] = None, copy_stream: Optional[torch.cuda.Stream] = None,
                 n_threads: int = 0) -> "Prefetched":
        """Start fetching the rows of a prefill batch.

        The hash runs on the current stream (a few microseconds: enqueue it
        ahead of the work the fetch should overlap, since it needs SMs).  With
        a pinned host table the rest runs on ``copy_stream``: the row ids go to
        the host, ``n_threads`` host threads gather the 264-byte rows into a
        pinned staging buffer, one DMA moves it to the device and the rows are
        dequantised there (with block-FP8 weights: regrouped as stored for the
        FP8 projection).  With a device table the gather follows the hash on
        the current stream.  At most two batches may be waiting at a time.
        (E4M3 + E8M0 tables only.)
        """
        if self.row_dim is not None:
            raise ValueError("prefetch handles the 264-byte E4M3 + E8M0 row tables only")
        dev = raw_ids.device
        T = raw_ids.numel()
        slot = self._prefetch_slot(T, dev)
        cur = torch.cuda.current_stream(dev)
        cur.wait_event(slot["consumed"])
        engram_hash(self.layout, self.layer, raw_ids, cu_seqlens, self.token_map, hist, slot["rows"], slot["mask"],
                    status)
        ready = torch.cuda.Event()
        if self.table.is_cuda:
            if self.fp8:
                engram_gather_fp8(self.table, self.total_rows, slot["rows"], slot["e8"], slot["sf"], status)
            else:
                engram_gather_dequant(self.table, self.total_rows, slot["rows"], slot["e"], status)
            ready.record(cur)
        else:
            cs = copy_stream if copy_stream is not None else torch.cuda.Stream(dev)
            hashed = torch.cuda.Event()
            hashed.record(cur)
            cs.wait_event(hashed)
            with torch.cuda.stream(cs):
                slot["rows_h"].copy_(slot["rows"], non_blocking=True)
                engram_host_gather_async(self.table, self.total_rows, slot["rows_h"], slot["staging"], slot["bad"],
                                         cs, n_threads)
                slot["staged"].copy_(slot["staging"], non_blocking=True)
                if self.fp8:
                    engram_gather_fp8(slot["staged"], T * self.layout.n_cols, slot["staged_ids"], slot["e8"],
                                      slot["sf"], status)
                else:
                    engram_dequant_rows(slot["staged"], self.layout.n_cols, slot["e"], status)
                ready.record(cs)
        slot["busy"] = True
        return Prefetched(slot, T, ready, cu_seqlens)

    def prefill_prefetched(self, pf: "Prefetched", h: torch.Tensor, status: Optional[torch.Tensor] = None,
                           gate_out: Optional[torch.Tensor] = None, conv_state: Optional[tuple] = None):
        """The projection, gate and residual update of a prefetched batch on the
        current stream, after its rows are ready.  ``pf.bad_rows`` (host) holds
        the count of out-of-range row ids once this stream has passed it."""
        if not pf.slot["busy"]:
            raise EngramError("this prefetched batch was already consumed")
        dev = h.device
        cur = torch.cuda.current_stream(dev)
        cur.wait_event(pf.ready)
        b = dict(self._buffers(pf.T, dev))
        b.update(e=pf.slot["e"], e8=pf.slot["e8"], sf=pf.slot["sf"], mask=pf.slot["mask"], rows=pf.slot["rows"])
        self._gate(b, h, status, gate_out, cu_seqlens=pf.cu_seqlens, conv_state=conv_state)
        pf.slot["consumed"].record(cur)
        pf.slot["busy"] = False
        return b

    def decode_graph(self, batch: int, hist: torch.Tensor, h: torch.Tensor, status: Optional[torch.Tensor] = None,
                     gate_out: Optional[torch.Tensor] = None, conv_state: Optional[tuple] = None) -> "DecodeGraph":
        """The decode step for a fixed batch captured as a CUDA graph (see DecodeGraph)."""
        return DecodeGraph(self, batch, hist, h, status, gate_out, conv_state)

    def decode(self, raw_ids: torch.Tensor, slots: torch.Tensor, hist: torch.Tensor, h: torch.Tensor,
               status: Optional[torch.Tensor] = None, gate_out: Optional[torch.Tensor] = None,
               conv_state: Optional[tuple] = None):
        B = raw_ids.numel()
        b = self._buffers(B, raw_ids.device)
        if self.row_dim is not None:
            engram_hash_step(self.layout, self.layer, raw_ids, slots, self.token_map, hist, b["rows"], b["mask"],
                             status)
            engram_gather_rows_bf16(self.table, b["rows"], b["e"], status)
        elif self.fp8:
            engram_hash_gather_step_fp8(self.layout, self.layer, raw_ids, slots, self.token_map, self.table, hist,
                                        b["e8"], b["sf"], b["mask"], b["rows"], status)
        else:
            engram_hash_gather_step(self.layout, self.layer, raw_ids, slots, self.token_map, self.table, hist,
                                    b["e"], b["mask"], b["rows"], status)
        self._gate(b, h, status, gate_out, slots=slots, conv_state=conv_state)
        return b

    def _gate(self, b, h, status, gate_out, cu_seqlens=None, slots=None, conv_state=None):
        if self.conv is not None:
            # the original layer: gates, then the short convolution with the residual add
            c = self.conv
            T = h.shape[0]
            self._project(b, h, status)
            g = engram_gates(b["partials"], T, self.hidden, self.hc, b["mask"], self.eps, self.clamp,
                             self.score_scale, gate_out if gate_out is not None else b["gate"])
            state, head = conv_state if conv_state is not None else (None, None)
            engram_short_conv_add(g, b["v"], h, b["mask"], c.w, c.gamma, c.dilation, c.eps, cu_seqlens,
                                  slots if cu_seqlens is None else None, state, head, b["conv_ws"], status)
            return
        if self.fused and self.fp8:
            engram_project_gate_fp8(b["e8"], b["sf"], self.w8p, self.sfb, h, self.q_w, self.k_w, b["mask"], self.eps,
                                    self.clamp, self.score_scale, gate_out, b["work"], status)
        elif self.fused:
            engram_project_gate(b["e"], self.wkv_packed, h, self.q_w, self.k_w, b["mask"], self.eps, self.clamp,
                                self.score_scale, gate_out, b["work"], status)
        else:
            self._project(b, h, status)
            engram_gate_add(b["partials"], b["v"], h, b["mask"], self.eps, self.clamp, self.score_scale, gate_out)

    def _project(self, b, h, status):
        """The unfused projection: partial sums and bf16 v into the layer's buffers."""
        if self.fp8:
            engram_project_fp8(b["e8"], b["sf"], self.w8p, self.sfb, h, self.q_w, self.k_w, b["partials"], b["v"],
                               status)
        else:
            engram_project(b["e"], self.wkv_packed, h, self.q_w, self.k_w, b["partials"], b["v"], status)


class DecodeGraph:
    """One decode step of a layer, for a fixed batch, captured as a CUDA graph.

    Write the step's raw ids (and the slots, when they change) into
    ``raw_ids`` / ``slots`` in place, then ``replay()``: the same kernels as
    ``EngramLayer.decode`` run on the current stream without any host-side
    launch work.  ``hist``, ``h``, ``status``, ``gate_out`` and the
    short-convolution state are the tensors given here; the step updates
    them in place exactly as ``decode`` does.  The graph keeps the layer's
    work buffers for this batch size alive for its own lifetime.
    """

    def __init__(self, layer: "EngramLayer", batch: int, hist: torch.Tensor, h: torch.Tensor,
                 status: Optional[torch.Tensor] = None, gate_out: Optional[torch.Tensor] = None,
                 conv_state: Optional[tuple] = None):
        dev = h.device
        self.raw_ids = torch.zeros(batch, dtype=torch.int32, device=dev)
        self.slots = torch.arange(batch, dtype=torch.int32, device=dev)
        self.hist, self.h, self.status, self.gate_out, self.conv_state = hist, h, status, gate_out, conv_state
        self.buffers = layer._buffers(batch, dev)
        _load()
        self.graph = torch.cuda.CUDAGraph()
        # capture records the launches only: hist and h are not touched here
        with torch.cuda.graph(self.graph):
            layer.decode(self.raw_ids, self.slots, hist, h, status, gate_out, conv_state)

    def replay(self):
        self.graph.replay()


class ShortConv:
    """Filters of the original Engram layer's short convolution: w f32
    [K][hc][H] (w[k] multiplies the value k*dilation positions back), RMSNorm
    weight gamma f32 [hc][H], dilation (the pages use the largest n-gram
    order) and the RMSNorm eps."""

    def __init__(self, w: torch.Tensor, gamma: torch.Tensor, dilation: int, eps: float = 1e-6):
        self.w, self.gamma, self.dilation, self.eps = w, gamma, dilation, eps


class Prefetched:
    """A batch whose rows are being fetched by ``EngramLayer.prefetch``."""

    def __init__(self, slot: dict, T: int, ready: torch.cuda.Event, cu_seqlens: torch.Tensor):
        self.slot, self.T, self.ready, self.cu_seqlens = slot, T, ready, cu_seqlens

    @property
    def e(self) -> torch.Tensor:
        return self.slot["e"]

    @property
    def mask(self) -> torch.Tensor:
        return self.slot["mask"]

    @property
    def row_ids(self) -> torch.Tensor:
        return self.slot["rows"]

    @property
    def bad_rows(self) -> int:
        return int(self.slot["bad"].item())
