"""Python binding of libqp, the GB300 Code Predictor library.

Argument marshalling only: every step of the frame loop runs in the CUDA
kernels of ``libqp.so`` behind the C ABI declared in ``include/qp.h``.
Importing this package loads the library and fails loudly if it has not
been built (``codebook_rvq_code_gb300.build.build()``); there is no CPU path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

from .build import LIB_PATH

QP_OK = 0
STATUS_NAMES = {
    0: "QP_OK", 1: "QP_ERR_ARG", 2: "QP_ERR_STATE", 3: "QP_ERR_WEIGHT_MISSING", 4: "QP_ERR_WEIGHT_SHAPE",
    5: "QP_ERR_WEIGHT_DTYPE", 6: "QP_ERR_CUDA", 7: "QP_ERR_TIMEOUT", 8: "QP_ERR_BAD_TOKEN", 9: "QP_ERR_OOM",
    10: "QP_ERR_UNKNOWN_WEIGHT", 11: "QP_ERR_DUPLICATE_WEIGHT",
}
DTYPES = {"bf16": 0, "f16": 1, "f32": 2, "q8_0": 3}

# every symbol include/qp.h declares
EXPORTED = [
    "qp_abi_version", "qp_status_string", "qp_default_geometry", "qp_create", "qp_load_weights",
    "qp_predict_frames", "qp_predict_frames_ex", "qp_predict_frames_host", "qp_get_device_status",
    "qp_launches_per_call", "qp_destroy", "qp_predict_frames_static", "qp_code_embeddings",
    "qp_set_deterministic",
    "qp_set_engine", "qp_trace_enable", "qp_trace_read", "qp_debug_waits",   # include/qp_debug.h
    "qp_rvq_normalize", "qp_rvq_decode",                   # include/qp_rvq.h
    "qp_gguf_open", "qp_gguf_close", "qp_gguf_tensor_count", "qp_gguf_tensor_info",   # include/qp_gguf.h
    "qp_gguf_geometry", "qp_gguf_load_weights",
    "qp_begin_frames", "qp_step_frames", "qp_begin_frames_ex", "qp_step_frames_ex",   # include/qp_sched.h
]


class QpGeometry(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("hidden", "layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn",
                                             "vocab", "n_steps", "talker_hidden", "code_embed_dim", "q0_vocab")] + \
               [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)]


class QpWeight(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("dtype", ctypes.c_int), ("dev_ptr", ctypes.c_void_p),
                ("shape", ctypes.c_int64 * 2)]


class QpSampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int), ("gumbel", ctypes.c_void_p)]


class QpError(RuntimeError):
    def __init__(self, where: str, code: int):
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")
        self.code = code


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libqp.so not built at {path}; run codebook_rvq_code_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, cp = ctypes.c_void_p, ctypes.c_int, ctypes.c_char_p
    lib.qp_abi_version.restype = i32
    lib.qp_status_string.restype = cp
    lib.qp_status_string.argtypes = [i32]
    lib.qp_default_geometry.restype = i32
    lib.qp_default_geometry.argtypes = [ctypes.POINTER(QpGeometry)]
    lib.qp_create.restype = i32
    lib.qp_create.argtypes = [ctypes.POINTER(QpGeometry), i32, ctypes.POINTER(vp)]
    lib.qp_load_weights.restype = i32
    lib.qp_load_weights.argtypes = [vp, ctypes.POINTER(QpWeight), i32, vp]
    lib.qp_predict_frames.restype = i32
    lib.qp_predict_frames.argtypes = [vp, i32, vp, vp, vp, vp, vp]
    lib.qp_predict_frames_ex.restype = i32
    lib.qp_predict_frames_ex.argtypes = [vp, i32, vp, vp, vp, vp, ctypes.POINTER(QpSampling), vp, vp]
    lib.qp_predict_frames_host.restype = i32
    lib.qp_predict_frames_host.argtypes = [vp, i32, vp, vp, vp, ctypes.POINTER(QpSampling), vp]
    lib.qp_predict_frames_static.restype = i32
    lib.qp_predict_frames_static.argtypes = [vp, i32, vp, vp, vp, vp, vp]
    lib.qp_get_device_status.restype = i32
    lib.qp_get_device_status.argtypes = [vp, vp]
    lib.qp_launches_per_call.restype = i32
    lib.qp_launches_per_call.argtypes = [vp, i32, i32]
    lib.qp_code_embeddings.restype = i32
    lib.qp_code_embeddings.argtypes = [vp, i32, vp, vp, vp]
    lib.qp_destroy.restype = None
    lib.qp_destroy.argtypes = [vp]
    lib.qp_set_engine.restype = i32
    lib.qp_set_engine.argtypes = [vp, i32]
    lib.qp_set_deterministic.restype = i32
    lib.qp_set_deterministic.argtypes = [vp, i32]
    lib.qp_debug_waits.restype = i32
    lib.qp_debug_waits.argtypes = [vp, i32, i32]
    lib.qp_trace_enable.restype = i32
    lib.qp_trace_enable.argtypes = [vp, i32]
    lib.qp_trace_read.restype = i32
    lib.qp_trace_read.argtypes = [vp, vp, i32, ctypes.POINTER(ctypes.c_int)]
    lib.qp_rvq_normalize.restype = i32
    lib.qp_rvq_normalize.argtypes = [vp, vp, i32, i32, i32, vp, vp]
    lib.qp_rvq_decode.restype = i32
    lib.qp_rvq_decode.argtypes = [vp, i32, i32, i32, vp, i32, vp, vp, vp]
    lib.qp_gguf_open.restype = i32
    lib.qp_gguf_open.argtypes = [ctypes.c_char_p, ctypes.POINTER(vp)]
    lib.qp_gguf_close.restype = None
    lib.qp_gguf_close.argtypes = [vp]
    lib.qp_gguf_tensor_count.restype = i32
    lib.qp_gguf_tensor_count.argtypes = [vp]
    lib.qp_gguf_tensor_info.restype = i32
    lib.qp_gguf_tensor_info.argtypes = [vp, i32, ctypes.POINTER(cp), ctypes.POINTER(ctypes.c_int),
                                        ctypes.POINTER(ctypes.c_int64)]
    lib.qp_gguf_geometry.restype = i32
    lib.qp_gguf_geometry.argtypes = [vp, vp, ctypes.POINTER(QpGeometry)]
    lib.qp_gguf_load_weights.restype = i32
    lib.qp_gguf_load_weights.argtypes = [vp, ctypes.POINTER(vp), i32, vp]
    lib.qp_begin_frames.restype = i32
    lib.qp_begin_frames.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp]
    lib.qp_step_frames.restype = i32
    lib.qp_step_frames.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp]
    lib.qp_begin_frames_ex.restype = i32
    lib.qp_begin_frames_ex.argtypes = [vp, i32, vp, vp, vp, vp, vp, ctypes.POINTER(QpSampling), vp]
    lib.qp_step_frames_ex.restype = i32
    lib.qp_step_frames_ex.argtypes = [vp, i32, vp, vp, vp, vp, vp, ctypes.POINTER(QpSampling), vp]
    return lib


_LIB: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = load_library()
    return _LIB


class GgufFile:
    """A parsed GGUF file (qp_gguf_open): its tensor table and metadata stay
    on the host until a CodePredictor loads weights from it."""

    def __init__(self, path: str):
        self._lib = lib()
        self._f = vp_t()
        _check("qp_gguf_open", self._lib.qp_gguf_open(str(path).encode(), ctypes.byref(self._f)))
        self.path = str(path)

    def tensors(self):
        """[(name, dtype tag or None, (out, in))] in file order (HF shapes)."""
        out = []
        names = {v: k for k, v in DTYPES.items()}
        for i in range(self._lib.qp_gguf_tensor_count(self._f)):
            name = ctypes.c_char_p()
            dt = ctypes.c_int()
            shape = (ctypes.c_int64 * 2)()
            _check("qp_gguf_tensor_info", self._lib.qp_gguf_tensor_info(self._f, i, ctypes.byref(name),
                                                                        ctypes.byref(dt), shape))
            out.append((name.value.decode(), names.get(dt.value), (int(shape[0]), int(shape[1]))))
        return out

    def geometry(self, talker: "Optional[GgufFile]" = None) -> QpGeometry:
        """Predictor geometry from this file's keys and tensor shapes; the q0
        table may come from the Talker's file (qp_gguf_geometry)."""
        g = QpGeometry()
        _check("qp_gguf_geometry", self._lib.qp_gguf_geometry(self._f, talker._f if talker else None,
                                                                ctypes.byref(g)))
        return g

    def close(self):
        if getattr(self, "_f", None):
            self._lib.qp_gguf_close(self._f)
            self._f = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


vp_t = ctypes.c_void_p


def default_geometry() -> QpGeometry:
    g = QpGeometry()
    _check("qp_default_geometry", lib().qp_default_geometry(ctypes.byref(g)))
    return g


def geometry_from(obj) -> QpGeometry:
    """A QpGeometry from any object with the same field names."""
    g = QpGeometry()
    for name, _ in QpGeometry._fields_:
        setattr(g, name, getattr(obj, name))
    return g


def _check(where: str, code: int):
    if code != QP_OK:
        raise QpError(where, code)


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _stream_ptr(stream) -> Optional[int]:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream) or None


def rvq_normalize(embedding_sum, cluster_usage, out=None, stream=None):
    """EMA codebooks -> codebooks (include/qp_rvq.h): f32 CUDA tensors
    [Q, K, D] and [Q, K]; returns the [Q, K, D] codebooks."""
    import torch
    Q, K, D = (int(x) for x in embedding_sum.shape)
    if out is None:
        out = torch.empty_like(embedding_sum)
    _check("qp_rvq_normalize", lib().qp_rvq_normalize(_ptr(embedding_sum), _ptr(cluster_usage), Q, K, D, _ptr(out),
                                                      _stream_ptr(stream)))
    return out


def rvq_decode(codebooks, codes, out=None, status=None, stream=None):
    """sum_i codebooks[i][codes[:, i]] (include/qp_rvq.h): f32 [Q, K, D] and
    int32 [N, Q] CUDA tensors; returns the [N, D] sums."""
    import torch
    Q, K, D = (int(x) for x in codebooks.shape)
    N = int(codes.shape[0])
    if out is None:
        out = torch.empty((N, D), dtype=torch.float32, device=codebooks.device)
    _check("qp_rvq_decode", lib().qp_rvq_decode(_ptr(codebooks), Q, K, D, _ptr(codes), N, _ptr(out), _ptr(status),
                                                _stream_ptr(stream)))
    return out


class CodePredictor:
    """One qp_handle: weights plus scratch for batches of up to max_batch frames."""

    def __init__(self, geometry=None, max_batch: int = 1):
        self._lib = lib()
        self.geometry = default_geometry() if geometry is None else (
            geometry if isinstance(geometry, QpGeometry) else geometry_from(geometry))
        self.max_batch = max_batch
        h = ctypes.c_void_p()
        _check("qp_create", self._lib.qp_create(ctypes.byref(self.geometry), max_batch, ctypes.byref(h)))
        self._h = h
        self._keep = []

    # -- weights -------------------------------------------------------------
    def load_weights(self, tensors: Dict[str, tuple], stream=None):
        """tensors: name -> (dtype tag, device tensor, shape); see qp_weight."""
        arr = (QpWeight * len(tensors))()
        names = []
        for i, (name, (dt, t, shape)) in enumerate(tensors.items()):
            nb = name.encode()
            names.append(nb)
            arr[i].name = nb
            arr[i].dtype = DTYPES[dt]
            arr[i].dev_ptr = int(t.data_ptr())
            arr[i].shape[0] = int(shape[0])
            arr[i].shape[1] = int(shape[1]) if len(shape) > 1 else 0
        _check("qp_load_weights", self._lib.qp_load_weights(self._h, arr, len(tensors), _stream_ptr(stream)))

    def load_raw_weights(self, raw, device="cuda", stream=None):
        """Upload storage-format tensors (objects with .name .dtype .shape .data
        numpy arrays) and hand them to qp_load_weights."""
        import torch
        up = {}
        for name, t in raw.items():
            data = torch.from_numpy(t.data.view("uint8").reshape(-1).copy()).to(device)
            up[name] = (t.dtype, data, t.shape)
        self.load_weights(up, stream=stream)
        torch.cuda.synchronize()
        return up

    # -- prediction ----------------------------------------------------------
    def predict(self, H, q0, out_codes=None, out_logits=None, sampling=None, forced=None, stream=None):
        """H [B, talker_hidden] f32 cuda, q0 [B] int32 cuda.  sampling: None
        or (temperature, top_k, gumbel [B, n_steps, vocab] f32 cuda).
        Returns out_codes [B, n_steps] int32 (allocated if not given)."""
        import torch
        B = int(H.shape[0])
        n = self.geometry.n_steps
        if out_codes is None:
            out_codes = torch.empty((B, n), dtype=torch.int32, device=H.device)
        samp = None
        if sampling is not None:
            T, k, gum = sampling
            samp = QpSampling(float(T), int(k), _ptr(gum))
        _check("qp_predict_frames_ex", self._lib.qp_predict_frames_ex(
            self._h, B, _ptr(H), _ptr(q0), _ptr(out_codes), _ptr(out_logits),
            ctypes.byref(samp) if samp is not None else None, _ptr(forced), _stream_ptr(stream)))
        return out_codes

    def predict_host(self, H_host, q0_host, codes_host, sampling=None, stream=None):
        """Host buffers (numpy or CPU tensors): copies in, predicts, copies the
        codes back and synchronises, all inside the library call."""
        samp = None
        if sampling is not None:
            T, k, gum = sampling
            samp = QpSampling(float(T), int(k), _ptr(gum))

        def hp(a):
            return a.ctypes.data if hasattr(a, "ctypes") else int(a.data_ptr())
        B = int(H_host.shape[0])
        _check("qp_predict_frames_host", self._lib.qp_predict_frames_host(
            self._h, B, hp(H_host), hp(q0_host), hp(codes_host),
            ctypes.byref(samp) if samp is not None else None, _stream_ptr(stream)))
        return codes_host

    def predict_static(self, H, q0, out_codes=None, out_logits=None, stream=None):
        """Greedy prediction through qp_predict_frames_static (scratch in the
        library's static device array; B <= 8)."""
        import torch
        B = int(H.shape[0])
        if out_codes is None:
            out_codes = torch.empty((B, self.geometry.n_steps), dtype=torch.int32, device=H.device)
        _check("qp_predict_frames_static", self._lib.qp_predict_frames_static(
            self._h, B, _ptr(H), _ptr(q0), _ptr(out_codes), _ptr(out_logits), _stream_ptr(stream)))
        return out_codes

    # -- state-slot calls (include/qp_sched.h) --------------------------------
    @staticmethod
    def _host_i32(a):
        import numpy as np
        return np.ascontiguousarray(np.asarray(a, dtype=np.int32))

    @staticmethod
    def _sampling(sampling):
        if sampling is None:
            return None
        T, k, gum = sampling
        return QpSampling(float(T), int(k), _ptr(gum))

    def begin_frames(self, slots, H, q0, out_q1=None, out_logits=None, sampling=None, stream=None):
        """Step 1 of new frames into state slots: slots host ints [B], H
        [B, talker_hidden] f32 cuda, q0 [B] int32 cuda.  Returns q1 [B] int32
        cuda; out_logits, if given, is [B, vocab] f32 cuda.  sampling: None
        (greedy) or (temperature, top_k, gumbel [B, vocab] f32 cuda)."""
        import torch
        sl = self._host_i32(slots)
        B = int(sl.shape[0])
        if out_q1 is None:
            out_q1 = torch.empty((B,), dtype=torch.int32, device=H.device)
        samp = self._sampling(sampling)
        _check("qp_begin_frames_ex", self._lib.qp_begin_frames_ex(
            self._h, B, sl.ctypes.data, _ptr(H), _ptr(q0), _ptr(out_q1), _ptr(out_logits),
            ctypes.byref(samp) if samp is not None else None, _stream_ptr(stream)))
        return out_q1

    def step_frames(self, slots, steps, codes_in, out_codes=None, out_logits=None, sampling=None, stream=None):
        """One step for each row: slots and steps host ints [B] (steps in
        2..n_steps), codes_in [B] int32 cuda (q_{step-1} of each row).
        Returns the step's codes [B] int32 cuda; out_logits, if given, is
        [B, vocab] f32 cuda.  sampling as for begin_frames (each row's noise
        for its own step)."""
        import torch
        sl, st = self._host_i32(slots), self._host_i32(steps)
        B = int(sl.shape[0])
        if st.shape[0] != B:
            raise ValueError("slots and steps differ in length")
        if out_codes is None:
            out_codes = torch.empty((B,), dtype=torch.int32, device=codes_in.device)
        samp = self._sampling(sampling)
        _check("qp_step_frames_ex", self._lib.qp_step_frames_ex(
            self._h, B, sl.ctypes.data, st.ctypes.data, _ptr(codes_in), _ptr(out_codes), _ptr(out_logits),
            ctypes.byref(samp) if samp is not None else None, _stream_ptr(stream)))
        return out_codes

    def code_embeddings(self, codes, out=None, stream=None):
        """E_j[codes[:, j]] for j < n_steps as f32 [B, n_steps, code_embed_dim]
        (qp_code_embeddings): the frame's residual codes in the predictor's
        embedding space."""
        import torch
        B = int(codes.shape[0])
        g = self.geometry
        if out is None:
            out = torch.empty((B, g.n_steps, g.code_embed_dim), dtype=torch.float32, device=codes.device)
        _check("qp_code_embeddings", self._lib.qp_code_embeddings(self._h, B, _ptr(codes), _ptr(out),
                                                                  _stream_ptr(stream)))
        return out

    ENGINES = {"auto": 0, "tile": 1, "small": 2, "cluster": 3}

    def set_engine(self, engine: str):
        """Schedule for later calls (include/qp_debug.h): "auto", "tile",
        "small" or "cluster"."""
        _check("qp_set_engine", self._lib.qp_set_engine(self._h, self.ENGINES[engine]))

    def set_deterministic(self, on: bool = True):
        """Bit-identical results run to run (include/qp.h, qp_set_deterministic)."""
        _check("qp_set_deterministic", self._lib.qp_set_deterministic(self._h, int(bool(on))))

    def debug_waits(self, wait_limit_us: int = 0, withhold_gemm: int = -1):
        """Wait limit and withheld count of include/qp_debug.h (testing the
        device-side failure path)."""
        _check("qp_debug_waits", self._lib.qp_debug_waits(self._h, int(wait_limit_us), int(withhold_gemm)))

    def trace(self, enable: bool = True):
        """Turn the phase trace of include/qp_debug.h on or off."""
        _check("qp_trace_enable", self._lib.qp_trace_enable(self._h, int(enable)))

    def read_trace(self, phases: int):
        """The last call's stamps as a numpy array [phases, n_cta, 2] (ns)."""
        import numpy as np
        n_sm = ctypes.c_int(0)
        buf = np.zeros(phases * 1024 * 2, dtype=np.uint64)
        got = self._lib.qp_trace_read(self._h, buf.ctypes.data, phases, ctypes.byref(n_sm))
        if got < 0:
            raise QpError("qp_trace_read", QP_ERR_STATE)
        return buf[: got * n_sm.value * 2].reshape(got, n_sm.value, 2)

    def device_status(self, stream=None) -> int:
        return int(self._lib.qp_get_device_status(self._h, _stream_ptr(stream)))

    def launches_per_call(self, B: int, sampling: bool = False) -> int:
        return int(self._lib.qp_launches_per_call(self._h, B, int(sampling)))

    def load_gguf(self, *files, stream=None):
        """Load the predictor's tensors from GgufFile objects or paths
        (predictor file first, then the Talker's for the q0 table)."""
        opened = [f if isinstance(f, GgufFile) else GgufFile(f) for f in files]
        arr = (vp_t * len(opened))(*[f._f for f in opened])
        _check("qp_gguf_load_weights", self._lib.qp_gguf_load_weights(self._h, arr, len(opened),
                                                                      _stream_ptr(stream)))

    def close(self):
        if getattr(self, "_h", None):
            self._lib.qp_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
