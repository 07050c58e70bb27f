"""ctypes binding of the C ABI in include/tf.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libtf_dualar.so"

TF_OK = 0
STATUS = {0: "TF_OK", 1: "TF_E_INVAL", 2: "TF_E_NOMEM", 3: "TF_E_CUDA", 4: "TF_E_STATE",
          5: "TF_E_CAPACITY", 6: "TF_E_TIMEOUT", 7: "TF_E_NUMERIC"}
TF_WEIGHT_BF16, TF_WEIGHT_FP8, TF_WEIGHT_NVFP4 = 0, 1, 2
TF_DTYPE_BF16, TF_DTYPE_FP8_E4M3, TF_DTYPE_NVFP4 = 0, 1, 2
TF_FLAG_QK_NORM, TF_FLAG_QK_NORM_FAST, TF_FLAG_SLOW_CB_SUM, TF_FLAG_PAGED_KV = 1, 2, 4, 8


class TfConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "slow_layers", "fast_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "ffn",
        "text_vocab", "semantic_vocab", "n_codebooks", "codebook_size", "max_seq_len",
        "max_batch")] + [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                         ("weight_dtype", ctypes.c_int32), ("flags", ctypes.c_int32)]


class TfTensor(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 3), ("data", ctypes.c_void_p),
                ("row_scale", ctypes.c_void_p)]


class TfSampling(ctypes.Structure):
    _fields_ = [("top_k", ctypes.c_int32), ("temperature", ctypes.c_float),
                ("seed", ctypes.c_uint64), ("top_p", ctypes.c_float),
                ("rep_penalty", ctypes.c_float), ("rep_window", ctypes.c_int32)]


class TfInfo(ctypes.Structure):
    _fields_ = [("position", ctypes.c_int32), ("frame_index", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("graph_nodes", ctypes.c_int32),
                ("weight_bytes", ctypes.c_int64), ("frame_weight_bytes", ctypes.c_int64),
                ("device_bytes", ctypes.c_int64)]


EXPORTS = {
    # name: (restype, argtypes)
    "tf_create": (ctypes.c_int, [ctypes.POINTER(TfConfig), ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)]),
    "tf_load_weights": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(TfTensor), ctypes.c_int32]),
    "tf_prefill": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.POINTER(TfSampling), ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_void_p]),
    "tf_decode_frame": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(TfSampling), ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p]),
    "tf_decode_frames": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(TfSampling), ctypes.c_int32,
                                        ctypes.c_void_p]),
    "tf_set_stream": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "tf_get_stream": (ctypes.c_void_p, [ctypes.c_void_p]),
    "tf_get_info": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(TfInfo)]),
    "tf_last_error": (ctypes.c_char_p, [ctypes.c_void_p]),
    "tf_destroy": (None, [ctypes.c_void_p]),
    "tf_profile_kernel": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.POINTER(ctypes.c_float),
                                         ctypes.POINTER(ctypes.c_int64)]),
    "tf_prefill_seq": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32]),
    "tf_release_seq": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    "tf_test_inject": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    "tf_test_fail_alloc": (None, [ctypes.c_int32]),
    "tf_op_quantize_fp8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "tf_op_quantize_nvfp4": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "tf_op_select": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                    ctypes.POINTER(TfSampling), ctypes.c_int32, ctypes.c_int32,
                                    ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                                    ctypes.c_void_p, ctypes.c_void_p]),
    "tf_op_attention": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]),
    "tf_op_attention_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                               ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                               ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]),
    "tf_op_attention_prompt": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_void_p, ctypes.c_void_p]),
    "tf_op_gemm": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]),
    "tf_op_gemm_skinny": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                         ctypes.c_void_p]),
    "tf_op_gemm_skinny_fp8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_void_p, ctypes.c_void_p]),
    "tf_op_gemm_skinny_nvfp4": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                               ctypes.c_void_p, ctypes.c_void_p]),
    "tf_op_gemv": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                                  ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                  ctypes.POINTER(ctypes.c_float), ctypes.c_void_p]),
}

_LIB = None


def library_path() -> str:
    return os.path.join(HERE, LIB_NAME)


def lib() -> ctypes.CDLL:
    """Load libtf_dualar.so (built by __graft_entry__.build()); raise if absent."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{LIB_NAME} is not built; run __graft_entry__.build() first")
        L = ctypes.CDLL(path)
        for name, (res, args) in EXPORTS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


class TfError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


def _check(status: int, ctx=None):
    if status != TF_OK:
        msg = lib().tf_last_error(ctx)
        raise TfError(status, msg.decode() if msg else "")


def config_from_dims(d, weight_dtype: str = "bf16", max_batch: int = 1) -> TfConfig:
    return TfConfig(d.slow_layers, d.fast_layers, d.hidden, d.n_heads, d.n_kv_heads, d.head_dim,
                    d.ffn, d.text_vocab, d.semantic_vocab, d.n_codebooks, d.codebook_size,
                    d.max_seq_len, max_batch, d.rms_eps, d.rope_theta,
                    {"bf16": TF_WEIGHT_BF16, "fp8": TF_WEIGHT_FP8, "nvfp4": TF_WEIGHT_NVFP4}[weight_dtype],
                    (TF_FLAG_QK_NORM if getattr(d, "qk_norm", False) else 0)
                    | (TF_FLAG_QK_NORM_FAST if getattr(d, "qk_norm_fast", False) else 0)
                    | (TF_FLAG_SLOW_CB_SUM if getattr(d, "slow_cb_sum", False) else 0))


def _sampling(s) -> TfSampling:
    if s is None:
        return TfSampling(0, 1.0, 0, 1.0, 1.0, 0)
    return TfSampling(int(s.get("top_k", 0)), float(s.get("temperature", 1.0)),
                      int(s.get("seed", 0)) & 0xFFFFFFFFFFFFFFFF, float(s.get("top_p", 1.0)),
                      float(s.get("rep_penalty", 1.0)), int(s.get("rep_window", 0)))


def _ptr(a):
    """Data pointer of a contiguous numpy array or torch tensor (host or device)."""
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        assert a.flags["C_CONTIGUOUS"]
        return a.ctypes.data
    assert a.is_contiguous()
    return a.data_ptr()


class Decoder:
    """One decode context (tf_create ... tf_destroy)."""

    def __init__(self, dims, weight_dtype: str = "bf16", device: int = 0, max_batch: int = 1,
                 paged: bool = False):
        self.dims = dims
        self.cfg = config_from_dims(dims, weight_dtype, max_batch)
        if paged:
            self.cfg.flags |= TF_FLAG_PAGED_KV
        self.batch = 1  # sequences of the last prefill
        h = ctypes.c_void_p()
        _check(lib().tf_create(ctypes.byref(self.cfg), device, ctypes.byref(h)), None)
        self.h = h
        self.ncb = dims.n_codebooks
        self.vmax = max(dims.semantic_vocab, dims.codebook_size)

    def close(self):
        if self.h:
            lib().tf_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load_weights(self, tensors: dict, fp8: dict | None = None, batch: int = 64):
        """tensors: name -> bf16 bits (np.uint16 or torch int16/bfloat16 tensor, host or
        device).  fp8: optional name -> (codes uint8, scale float32) for linear weights."""
        keep = []
        items = []
        for name, arr in tensors.items():
            if fp8 and name in fp8:
                codes, scale = fp8[name]
                keep += [codes, scale]
                items.append(TfTensor(name.encode(), TF_DTYPE_FP8_E4M3, codes.ndim,
                                      (ctypes.c_int64 * 3)(*codes.shape, *([0] * (3 - codes.ndim))),
                                      _ptr(codes), _ptr(scale)))
            else:
                keep.append(arr)
                items.append(TfTensor(name.encode(), TF_DTYPE_BF16, arr.ndim,
                                      (ctypes.c_int64 * 3)(*arr.shape, *([0] * (3 - arr.ndim))),
                                      _ptr(arr), None))
        for s in range(0, len(items), batch):
            chunk = (TfTensor * len(items[s:s + batch]))(*items[s:s + batch])
            _check(lib().tf_load_weights(self.h, chunk, len(items[s:s + batch])), self.h)

    def prefill(self, tokens, sampling=None, forced=None, logits=False):
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        if tok.ndim == 1:
            tok = tok[None]
        frame = np.zeros((tok.shape[0], self.ncb), np.int32)
        lg = np.zeros((tok.shape[0], self.ncb, self.vmax), np.float32) if logits else None
        fo = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32)
        s = _sampling(sampling)
        _check(lib().tf_prefill(self.h, _ptr(tok), tok.shape[0], tok.shape[1], ctypes.byref(s),
                                _ptr(fo), _ptr(frame), _ptr(lg)), self.h)
        self.batch = tok.shape[0]
        self.active = set(range(tok.shape[0]))
        return frame, lg

    def prefill_seq(self, slot: int, tokens):
        """Start a sequence in `slot` (continuous batching); its frame 0 comes
        from the next decode call.  The batch becomes the slots up to the last
        active one."""
        tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
        _check(lib().tf_prefill_seq(self.h, slot, _ptr(tok), tok.size), self.h)
        self.active = getattr(self, "active", set()) | {slot}
        self.batch = max(self.active) + 1

    def release_seq(self, slot: int):
        _check(lib().tf_release_seq(self.h, slot), self.h)
        self.active = getattr(self, "active", set()) - {slot}
        self.batch = max(self.active) + 1 if self.active else 1

    def decode_frame(self, sampling=None, forced=None, logits=False):
        B = self.batch
        frame = np.zeros((B, self.ncb), np.int32)
        lg = np.zeros((B, self.ncb, self.vmax), np.float32) if logits else None
        fo = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32)
        s = _sampling(sampling)
        _check(lib().tf_decode_frame(self.h, ctypes.byref(s), _ptr(fo), _ptr(frame), _ptr(lg)),
               self.h)
        return frame, lg

    def decode_frames(self, n: int, sampling=None, out=None):
        frames = out if out is not None else np.zeros((n, self.batch, self.ncb), np.int32)
        s = _sampling(sampling)
        _check(lib().tf_decode_frames(self.h, ctypes.byref(s), n, _ptr(frames)), self.h)
        return frames

    def set_stream(self, stream_handle):
        _check(lib().tf_set_stream(self.h, ctypes.c_void_p(stream_handle)), self.h)

    def stream(self) -> int:
        return lib().tf_get_stream(self.h) or 0

    def profile_kernel(self, which: int, iters: int):
        """(ms per launch, algorithmic bytes per launch) of one in-frame kernel."""
        ms = ctypes.c_float(0.0)
        b = ctypes.c_int64(0)
        _check(lib().tf_profile_kernel(self.h, which, iters, ctypes.byref(ms), ctypes.byref(b)),
               self.h)
        return ms.value, b.value

    def info(self) -> dict:
        i = TfInfo()
        _check(lib().tf_get_info(self.h, ctypes.byref(i)), self.h)
        return {f: getattr(i, f) for f, _ in TfInfo._fields_}


def op_quantize_fp8(w_dev, rows, cols, codes_dev, scale_dev, stream=0):
    _check(lib().tf_op_quantize_fp8(w_dev, rows, cols, codes_dev, scale_dev, stream))


def op_quantize_nvfp4(w_dev, rows, cols, packed_dev, scale_dev, stream=0):
    _check(lib().tf_op_quantize_nvfp4(w_dev, rows, cols, packed_dev, scale_dev, stream))


def op_select(logits_dev, n, vocab, sampling, frame, codebook0, sequence, ids_dev, stream=0,
              recent_dev=None, n_recent=0):
    s = _sampling(sampling)
    _check(lib().tf_op_select(logits_dev, n, vocab, ctypes.byref(s), frame, codebook0, sequence,
                              recent_dev, n_recent, ids_dev, stream))


def op_attention(q_dev, K_dev, V_dev, T, Hq, Hkv, D, rows, pos0, splits, out_dev, stream=0):
    _check(lib().tf_op_attention(q_dev, K_dev, V_dev, T, Hq, Hkv, D, rows, pos0, splits, out_dev,
                                 stream))


def op_attention_prompt(q_dev, K_dev, V_dev, T, Hq, Hkv, D, rows, pos0, out_dev, stream=0):
    _check(lib().tf_op_attention_prompt(q_dev, K_dev, V_dev, T, Hq, Hkv, D, rows, pos0, out_dev,
                                        stream))


def op_gemm(A_dev, W_dev, M, N, K, C_dev, stream=0):
    _check(lib().tf_op_gemm(A_dev, W_dev, M, N, K, C_dev, stream))


def op_gemm_skinny(A_dev, W_dev, M, N, K, C_dev, stream=0):
    _check(lib().tf_op_gemm_skinny(A_dev, W_dev, M, N, K, C_dev, stream))


def op_gemm_skinny_fp8(A_dev, W_dev, scale_dev, M, N, K, C_dev, stream=0):
    _check(lib().tf_op_gemm_skinny_fp8(A_dev, W_dev, scale_dev, M, N, K, C_dev, stream))


def op_gemm_skinny_nvfp4(A_dev, W_dev, scale_dev, M, N, K, C_dev, stream=0):
    _check(lib().tf_op_gemm_skinny_nvfp4(A_dev, W_dev, scale_dev, M, N, K, C_dev, stream))


def op_gemv(W_dev, dtype, scale_dev, rows, cols, x_dev, y_dev, repeat=1, stream=0):
    ms = ctypes.c_float(0.0)
    _check(lib().tf_op_gemv(W_dev, dtype, scale_dev, rows, cols, x_dev, y_dev, repeat,
                            ctypes.byref(ms), stream))
    return ms.value
