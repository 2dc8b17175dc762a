"""Helpers for the GPU parity tests: move seeded numpy inputs to cuda:0, run
an entry point through the Python binding (which calls the C ABI), and bring
the bytes back for comparison with the CPU oracle."""
import numpy as np
import torch

DEV = torch.device("cuda:0")


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if not a.flags.writeable:
        a = a.copy()
    return torch.from_numpy(a).to(DEV)


def bf16_dev(a_u16: np.ndarray) -> torch.Tensor:
    """uint16 bit patterns -> CUDA bf16 tensor of the same shape (contiguous)."""
    return to_dev(np.ascontiguousarray(a_u16).view(np.int16)).view(torch.bfloat16)


def latent_dev(latent_view: np.ndarray) -> torch.Tensor:
    """A [T, d] uint16 view, possibly a column slice of a wider array: upload
    the whole underlying rows and slice on the device, so the row stride
    reaches the kernel."""
    stride = latent_view.strides[0] // 2
    T, d = latent_view.shape
    if stride == d:
        return bf16_dev(latent_view)
    base = np.lib.stride_tricks.as_strided(latent_view, shape=(T, stride),
                                           strides=latent_view.strides, writeable=False)
    return bf16_dev(np.ascontiguousarray(base))[:, :d]


def u16_host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def u8_host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().numpy()


def paged_cache_dev(buf: np.ndarray, offset: int, num_blocks: int, block_size: int,
                    block_stride_rows: int, pitch: int = 272):
    """Device copy of the whole buffer and the layer's [num_blocks,
    block_size, pitch] view at byte ``offset`` with block stride
    ``block_stride_rows`` rows."""
    d = to_dev(buf)
    if num_blocks == 1 and block_stride_rows == block_size:
        return d, d[offset:offset + block_size * pitch]
    view = d[offset:].as_strided((num_blocks, block_size, pitch),
                                 (block_stride_rows * pitch, pitch, 1))
    return d, view


def first_diff(got: np.ndarray, want: np.ndarray):
    bad = np.nonzero(got.reshape(-1) != want.reshape(-1))[0]
    if bad.size == 0:
        return None
    return f"{bad.size} differing bytes/elements; first at flat index {bad[:8].tolist()}"
