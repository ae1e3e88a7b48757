"""Write synthetic predictor weights as GGUF files (seeded test inputs).

The layout is the public GGUF version 3 container: header ("GGUF", version,
tensor count, metadata count), metadata key/values, the tensor table (name,
dimensions innermost first, GGML type, offset in the data section), then the
data, each tensor at a multiple of the alignment.  Tensor names, the F32 /
F16 / Q8_0 split and the qwen3-tts.code_pred.* geometry keys are those of the
exporter page ("rightkit-qts 0.2.3 - Qwen3-TTS 1.7B -> QTS GGUF", sections
"Loader contract" and "Upstream differences & verification scope").  This
module only serialises tensors from :mod:`synthetic`; it computes nothing of
the method.
"""
from __future__ import annotations

import struct
from typing import Dict, Iterable, Optional, Tuple

import numpy as np

GGML_TYPE = {"f32": 0, "f16": 1, "q8_0": 8, "bf16": 30}
# metadata value types
U32, I32, F32, STRING, ARRAY, U64 = 4, 5, 6, 8, 9, 10


def _str(s: str) -> bytes:
    b = s.encode()
    return struct.pack("<Q", len(b)) + b


def _value(vtype: int, v) -> bytes:
    if vtype == U32:
        return struct.pack("<I", int(v))
    if vtype == I32:
        return struct.pack("<i", int(v))
    if vtype == F32:
        return struct.pack("<f", float(v))
    if vtype == U64:
        return struct.pack("<Q", int(v))
    if vtype == STRING:
        return _str(str(v))
    if vtype == ARRAY:
        et, items = v
        return struct.pack("<IQ", et, len(items)) + b"".join(_value(et, x) for x in items)
    raise ValueError(vtype)


def predictor_metadata(g) -> Dict[str, Tuple[int, object]]:
    """The predictor file's geometry keys (and a few others a real file has)."""
    p = "qwen3-tts.code_pred."
    return {
        "general.architecture": (STRING, "qwen3-tts"),
        p + "embedding_length": (U32, g.hidden),
        p + "attention.key_length": (U32, g.head_dim),
        p + "attention.head_count": (U32, g.n_q_heads),
        p + "attention.head_count_kv": (U32, g.n_kv_heads),
        p + "feed_forward_length": (U32, g.ffn),
        p + "layer_count": (U32, g.layers),
        p + "vocab_size": (U32, g.vocab),
        p + "attention.layer_norm_rms_epsilon": (F32, g.rms_eps),
        p + "rope.freq_base": (F32, g.rope_theta),
        "tokenizer.ggml.tokens": (ARRAY, (STRING, ["<a>", "<b>", "<c>"])),
    }


def _blob(t) -> bytes:
    if t.dtype == "f16":
        return np.ascontiguousarray(t.data, dtype=np.float16).tobytes()
    if t.dtype == "bf16":
        return np.ascontiguousarray(t.data, dtype=np.uint16).tobytes()
    if t.dtype == "f32":
        return np.ascontiguousarray(t.data, dtype=np.float32).tobytes()
    if t.dtype == "q8_0":
        return np.ascontiguousarray(t.data, dtype=np.uint8).tobytes()
    raise ValueError(t.dtype)


def write_gguf(path: str, tensors: Iterable, metadata: Optional[Dict[str, Tuple[int, object]]] = None,
               alignment: int = 32, extra: Optional[Dict[str, np.ndarray]] = None) -> None:
    """tensors: RawTensor objects (HF shapes); extra: other f32 tensors a
    real file would hold (ignored by the predictor's loader)."""
    metadata = dict(metadata or {})
    if alignment != 32:
        metadata["general.alignment"] = (U32, alignment)
    items = []
    for t in tensors:
        items.append((t.name, tuple(reversed(t.shape)), GGML_TYPE[t.dtype], _blob(t)))
    for name, a in (extra or {}).items():
        a = np.ascontiguousarray(a, dtype=np.float32)
        items.append((name, tuple(reversed(a.shape)), GGML_TYPE["f32"], a.tobytes()))
    head = struct.pack("<IIQQ", 0x46554747, 3, len(items), len(metadata))
    for k, (vt, v) in metadata.items():
        head += _str(k) + struct.pack("<I", vt) + _value(vt, v)
    offsets, off = [], 0
    for _, _, _, blob in items:
        offsets.append(off)
        off = (off + len(blob) + alignment - 1) // alignment * alignment
    for (name, dims, ty, _), o in zip(items, offsets):
        head += _str(name) + struct.pack("<I", len(dims)) + b"".join(struct.pack("<Q", d) for d in dims)
        head += struct.pack("<IQ", ty, o)
    with open(path, "wb") as fh:
        fh.write(head)
        fh.write(b"\0" * ((-len(head)) % alignment))
        start = fh.tell()
        for (_, _, _, blob), o in zip(items, offsets):
            fh.write(b"\0" * (start + o - fh.tell()))
            fh.write(blob)


def write_predictor_files(pred_path: str, talker_path: str, g, raw, alignment: int = 32) -> None:
    """The exporter's split: code_pred.* in the predictor file with the
    geometry keys, the q0 table in the Talker's file among other tensors."""
    pred = [t for n, t in raw.items() if n.startswith("code_pred.")]
    write_gguf(pred_path, pred, predictor_metadata(g), alignment=alignment)
    write_gguf(talker_path, [raw["talker.codec_embd.weight"]],
               {"general.architecture": (STRING, "qwen3-tts")}, alignment=alignment,
               extra={"talker.output_norm.weight": np.ones(g.talker_hidden, np.float32)})
