"""ctypes binding of ``libtq.so`` (declared in ``include/tq.h``): the C entry points under their
own names, plus argument marshalling for torch tensors.  Every computation runs in the library's
CUDA kernels; nothing here computes.  Importing fails loudly when the library has not been built.
"""

import ctypes
import os

from . import _build

c_int32 = ctypes.c_int32
c_uint32 = ctypes.c_uint32
c_uint64 = ctypes.c_uint64
c_size_t = ctypes.c_size_t
c_void_p = ctypes.c_void_p

TQ_OK = 0
TQ_ERR_INVALID_ARG = 1
TQ_ERR_UNSUPPORTED = 2
TQ_ERR_CAPACITY = 3
TQ_ERR_WORKSPACE = 4
TQ_ERR_CUDA = 5
TQ_ERR_DEVICE = 6
TQ_ERR_STATE = 7

TQ_PLAIN_KV, TQ_TQ_KV, TQ_KQV, TQ_QKQV, TQ_SQU_KV = 0, 1, 2, 3, 4
TQ_F32, TQ_BF16, TQ_F16 = 0, 1, 2
TQ_MAX_BATCH = 512

SCHEMES = {"plain": TQ_PLAIN_KV, "plain-kv": TQ_PLAIN_KV, "kv": TQ_PLAIN_KV,
           "tq": TQ_TQ_KV, "tq-kv": TQ_TQ_KV, "kqv": TQ_KQV, "qkqv": TQ_QKQV, "tq-qkv": TQ_QKQV,
           "squ": TQ_SQU_KV, "squ-kv": TQ_SQU_KV}


class tq_codec(ctypes.Structure):
    _fields_ = [("bits", c_int32), ("rotate", c_int32), ("qjl", c_int32)]


class tq_config(ctypes.Structure):
    _fields_ = [("head_dim", c_int32), ("num_q_heads", c_int32), ("num_kv_heads", c_int32),
                ("batch", c_int32), ("capacity", c_int32), ("k", tq_codec), ("v", tq_codec),
                ("qjl_m", c_int32), ("headq_rank", c_int32), ("headq_bits", c_int32),
                ("seed", c_uint64)]


class tq_region(ctypes.Structure):
    _fields_ = [("offset", c_uint64), ("record_bytes", c_uint64)]


REGION_NAMES = ["k_codes", "k_norm", "k_signs", "k_rho", "k_side", "k_side_scale",
                "v_codes", "v_norm", "v_signs", "v_rho"]


class tq_cache_layout(ctypes.Structure):
    _fields_ = [("layout_version", c_uint32), ("tile_tokens", c_uint32), ("total_bytes", c_uint64),
                ("k_offset", c_uint64), ("k_block_bytes", c_uint64), ("v_offset", c_uint64),
                ("v_block_bytes", c_uint64)] + [(n, tq_region) for n in REGION_NAMES]


class tq_page_table(ctypes.Structure):
    _fields_ = [("block_table", c_void_p), ("max_blocks_per_seq", c_int32), ("num_pages", c_int32)]


TQ_DEVERR_WAIT_TIMEOUT = 1
TQ_DEVERR_SMEM_PLAN = 2
TQ_DEVERR_BAD_PAGE = 3
TQ_DEVERR_BAD_LENGTH = 4


class TQError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{message} (status {status})")
        self.status = status


def _load():
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    return ctypes.CDLL(path)


lib = _load()

# (name, restype, argtypes) of every entry point declared in include/tq.h
DECLARATIONS = [
    ("tq_config_from_scheme", c_int32, [c_int32, c_int32, ctypes.POINTER(tq_config)]),
    ("tq_context_create", c_int32, [ctypes.POINTER(tq_config), ctypes.POINTER(c_void_p)]),
    ("tq_context_destroy", None, [c_void_p]),
    ("tq_tables_bytes", c_size_t, [c_void_p]),
    ("tq_tables_host", c_int32, [c_void_p, c_void_p, c_size_t]),
    ("tq_tables_upload", c_int32, [c_void_p, c_void_p, c_void_p]),
    ("tq_headq_set_basis", c_int32, [c_void_p, c_void_p, c_void_p]),
    ("tq_spectral_set_basis", c_int32, [c_void_p, c_int32, c_void_p, c_void_p, c_void_p]),
    ("tq_get_cache_layout", c_int32, [c_void_p, ctypes.POINTER(tq_cache_layout)]),
    ("tq_quantize_append", c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32,
                                     ctypes.POINTER(c_int32), c_void_p]),
    ("tq_decode_workspace_bytes", c_size_t, [c_void_p, c_int32]),
    ("tq_decode_attention", c_int32, [c_void_p, c_void_p, c_void_p, ctypes.POINTER(c_int32), c_void_p,
                                      c_void_p, c_size_t, c_void_p]),
    ("tq_append_decode_attention", c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32,
                                             c_void_p, ctypes.POINTER(c_int32), c_void_p, c_void_p, c_size_t,
                                             c_void_p]),
    ("tq_prefill_workspace_bytes", c_size_t, [c_void_p, c_int32]),
    ("tq_prefill_attention", c_int32, [c_void_p, c_void_p, c_void_p, c_int32, ctypes.POINTER(c_int32),
                                       c_void_p, c_void_p, c_size_t, c_void_p]),
    ("tq_decode_attention_static", c_int32, [c_void_p, c_void_p, c_void_p, ctypes.POINTER(c_int32),
                                             c_void_p, c_void_p]),
    ("tq_decode_attention_multi", c_int32, [c_void_p, c_void_p, c_void_p, c_int32, ctypes.POINTER(c_int32),
                                            c_void_p, c_void_p, c_size_t, c_void_p]),
    ("tq_headq_correct", c_int32, [c_void_p, c_void_p, c_void_p, ctypes.POINTER(c_int32), c_void_p,
                                   c_int32, c_void_p]),
    ("tq_dequantize", c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_void_p,
                                c_void_p, c_void_p]),
    ("tq_get_paged_cache_layout", c_int32, [c_void_p, c_int32, ctypes.POINTER(tq_cache_layout)]),
    ("tq_quantize_append_paged", c_int32, [c_void_p, c_void_p, ctypes.POINTER(tq_page_table), c_void_p,
                                           c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p]),
    ("tq_decode_attention_paged", c_int32, [c_void_p, c_void_p, ctypes.POINTER(tq_page_table), c_void_p,
                                            c_int32, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    ("tq_get_device_error", c_int32, [c_void_p, ctypes.POINTER(c_int32), c_void_p]),
    ("tq_get_static_device_error", c_int32, [ctypes.POINTER(c_int32), c_void_p]),
    ("tq_status_string", ctypes.c_char_p, [c_int32]),
    ("tq_last_error", ctypes.c_char_p, []),
]

for _name, _res, _args in DECLARATIONS:
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args
    globals()[_name] = _fn


def check(status):
    """Raise TQError for a non-zero status, with the library's message."""
    if status != TQ_OK:
        msg = lib.tq_last_error().decode() or lib.tq_status_string(status).decode()
        raise TQError(status, msg)
    return status


def int_array(values):
    arr = (c_int32 * max(1, len(values)))()
    for i, v in enumerate(values):
        arr[i] = int(v)
    return arr
