"""Shared test helpers: dtype bit-casts between torch and numpy, e4m3
decoding through torch (a library routine independent of the oracle), and
the output comparison rule."""
import numpy as np
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    return bits_to_bf16(a).double().numpy()


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()


def row_rel_err(y: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per token row: max |y - ref| / max(max |ref|, 1e-6)."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.abs(y - ref).max(axis=1)
    den = np.maximum(np.abs(ref).max(axis=1), 1e-6)
    return num / den


def elem_rel_err(y: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Element-wise |y - ref| / max(|ref|, 1e-2 * rowmax |ref|) (reported
    beside the per-row bar)."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    rowmax = np.abs(ref).max(axis=1, keepdims=True)
    return np.abs(y - ref) / np.maximum(np.abs(ref), np.maximum(1e-2 * rowmax, 1e-30))
