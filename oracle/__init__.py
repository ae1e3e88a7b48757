"""CPU oracle of the Code Predictor loop -- TEST INFRASTRUCTURE, NOT THE PRODUCT.

Only the tests, the smoke check and bench.py's CPU-baseline / reference legs
may import this package.  It shares no code with the CUDA library.
"""
from .predictor import (Predictor, attend, bf16_to_f32, code_embeddings, dequant_q8_0, forward_sequence,
                        greedy_code, gumbel_topk_code, predict_frames,
                        predict_frames_bruteforce, quant_q8_0, rms_norm, rope,
                        rope_angles, round_to_f16, sampling_decidable, silu, top2_gap, topk_set,
                        weights_to_f32)
from .rvq import ema_codebook, rvq_decode, rvq_encode

__all__ = [n for n in dir() if not n.startswith("_")]
