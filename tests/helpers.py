"""Shared helpers of the GPU parity tests: tensor <-> numpy marshalling and
the GEMM tolerance. No method arithmetic lives here."""
import numpy as np
import torch

# GEMM tolerance: global relative Frobenius error and a per-element bound
# (bf16 output rounding is 2^-9 relative; 2^-7 leaves room for fp32
# accumulation-order differences; the rms term covers cancellation).
REL_FRO = 1e-3
ELEM_REL = 2.0 ** -7
ELEM_RMS = 1e-2


def np_input(t: torch.Tensor) -> np.ndarray:
    """CPU numpy view of a bf16 (as uint16 bits) or fp32 tensor, keeping strides."""
    t = t.cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def np_bytes(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.uint8).cpu().numpy()


def np_sf(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def check_gemm(got: np.ndarray, ref: np.ndarray, what: str = "gemm") -> float:
    got = got.astype(np.float64)
    err = got - ref
    den = np.linalg.norm(ref)
    rel = np.linalg.norm(err) / den if den > 0 else np.linalg.norm(err)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    bound = ELEM_REL * np.abs(ref) + ELEM_RMS * rms
    bad = np.abs(err) > bound
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3e} > {REL_FRO}"
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of tolerance; first at "
                           f"{np.argwhere(bad)[0]} got {got[bad][0]} ref {ref[bad][0]}")
    return rel
