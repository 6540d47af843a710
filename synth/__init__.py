"""Seeded synthetic inputs for the routed-MoE workloads (shared by the oracle side
and the GPU side; holds none of the method's arithmetic).

The C source `synth.c` is compiled on first use (or by `__graft_entry__.build()`)
into `synth/_build/libsynth.so` and driven through ctypes.  All values are
bit-identical across x86-64 and aarch64.

Workloads (sizes of the synthetic model; every value seeded with seed 0):

=================  ======  =====  ===  =====  ======  ======
name               hidden  exp.   k    inter  layers  tokens
=================  ======  =====  ===  =====  ======  ======
tiny               512     32     4    128    1       4
decode_layer       2048    512    10   512    1       1000
decode_stack       2048    512    10   512    48      256
prefill_chunk      2048    512    10   512    1       512
prefill_bounded    2048    512    10   512    48      2048
=================  ======  =====  ===  =====  ======  ======

`prefill_bounded` adds a Zipf(1.1) router bias and 435 of 512 experts resident
per layer.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None

TAG_GRID, TAG_ROUTER, TAG_QBLK, TAG_X, TAG_ZIPF, TAG_RESID, TAG_SLOTPERM = 1, 2, 3, 4, 5, 6, 7
BLOCK_VALUES = 256
BLOCK_BYTES = 66


@dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    n_layers: int
    tokens: int
    zipf_s: float = 0.0          # 0 = no router bias
    n_resident: int = -1         # -1 = every expert resident
    seed: int = 0

    @property
    def matrix_bytes(self) -> int:
        return self.hidden * self.inter // BLOCK_VALUES * BLOCK_BYTES

    @property
    def record_bytes(self) -> int:
        return 3 * self.matrix_bytes


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny", 512, 32, 4, 128, 1, 4),
        Workload("decode_layer", 2048, 512, 10, 512, 1, 1000),
        Workload("decode_stack", 2048, 512, 10, 512, 48, 256),
        Workload("prefill_chunk", 2048, 512, 10, 512, 1, 512),
        Workload("prefill_bounded", 2048, 512, 10, 512, 48, 2048, zipf_s=1.1, n_resident=435),
    )
}
# token streams of different workloads are decorrelated by this id
_TOKEN_STREAM = {"tiny": 1, "decode_layer": 2, "decode_stack": 3, "prefill_chunk": 4, "prefill_bounded": 5}


def build(force: bool = False) -> str:
    """Compile synth.c into _build/libsynth.so (gcc, -ffp-contract=off, OpenMP)."""
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    src = os.path.join(_HERE, "synth.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-Wall", "-Wextra", "-Werror", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            u64, u32, i32, i64, dbl, vp = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32,
                                           ctypes.c_int64, ctypes.c_double, ctypes.c_void_p)
            L.synth_mix64.restype = u64; L.synth_mix64.argtypes = [u64]
            L.synth_key.restype = u64; L.synth_key.argtypes = [u64, u32, u64, u64]
            L.synth_draw.restype = u64; L.synth_draw.argtypes = [u64, u64]
            L.synth_ln.restype = dbl; L.synth_ln.argtypes = [dbl]
            L.synth_sincos2pi.restype = None
            L.synth_sincos2pi.argtypes = [dbl, ctypes.POINTER(dbl), ctypes.POINTER(dbl)]
            L.synth_f16_bits.restype = ctypes.c_uint16; L.synth_f16_bits.argtypes = [dbl]
            L.synth_grid.restype = None; L.synth_grid.argtypes = [u64, vp]
            L.synth_matrix_blocks.restype = None
            L.synth_matrix_blocks.argtypes = [u64, i32, i32, i32, i64, vp]
            L.synth_expert_records.restype = None
            L.synth_expert_records.argtypes = [u64, i32, i32, i32, i32, i32, vp, i32]
            L.synth_normal_f32.restype = None
            L.synth_normal_f32.argtypes = [u64, u32, u64, u64, i64, dbl, vp, i32]
            L.synth_zipf_bias.restype = None
            L.synth_zipf_bias.argtypes = [u64, i32, i32, dbl, vp, vp]
            L.synth_resident_mask.restype = None
            L.synth_resident_mask.argtypes = [u64, i32, i32, i32, vp, vp]
            L.synth_permutation.restype = None
            L.synth_permutation.argtypes = [u64, u32, u64, i32, vp]
            _lib = L
    return _lib


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def grid(seed: int = 0) -> np.ndarray:
    """The 256 x 8 int8 codebook grid."""
    out = np.empty((256, 8), dtype=np.int8)
    lib().synth_grid(seed, out.ctypes.data)
    return out


def matrix_blocks(layer: int, expert: int, matrix: int, nblocks: int, seed: int = 0) -> np.ndarray:
    out = np.empty(nblocks * BLOCK_BYTES, dtype=np.uint8)
    lib().synth_matrix_blocks(seed, layer, expert, matrix, nblocks, out.ctypes.data)
    return out


def expert_records_into(ptr: int, w: Workload, layer: int, e0: int, n: int, nthreads: int = 0) -> None:
    """Write n consecutive expert records (experts e0..e0+n-1 of `layer`) at host address ptr."""
    lib().synth_expert_records(w.seed, layer, e0, n, w.hidden, w.inter, ptr, nthreads or _threads())


def expert_records(w: Workload, layer: int, e0: int = 0, n: int = 1, nthreads: int = 0) -> np.ndarray:
    out = np.empty((n, w.record_bytes), dtype=np.uint8)
    expert_records_into(out.ctypes.data, w, layer, e0, n, nthreads)
    return out


def normal_f32(tag: int, a: int, b: int, n: int, sigma: float, seed: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().synth_normal_f32(seed, tag, a, b, n, sigma, out.ctypes.data, _threads())
    return out


def router(w: Workload, layer: int) -> np.ndarray:
    """Router matrix W_r [E][H] f32 ~ N(0, 0.02^2)."""
    return normal_f32(TAG_ROUTER, layer, 0, w.n_experts * w.hidden, 0.02, w.seed).reshape(
        w.n_experts, w.hidden)


def tokens(w: Workload, t0: int = 0, n: int | None = None) -> np.ndarray:
    """Activations x [n][H] f32 ~ N(0, 1) for tokens t0..t0+n-1 of workload w."""
    n = w.tokens - t0 if n is None else n
    out = np.empty((n, w.hidden), dtype=np.float32)
    for i in range(n):
        out[i] = normal_f32(TAG_X, t0 + i, _TOKEN_STREAM[w.name], w.hidden, 1.0, w.seed)
    return out


def zipf_bias(w: Workload, layer: int) -> np.ndarray:
    out = np.empty(w.n_experts, dtype=np.float32)
    perm = np.empty(w.n_experts, dtype=np.int32)
    lib().synth_zipf_bias(w.seed, layer, w.n_experts, w.zipf_s, out.ctypes.data, perm.ctypes.data)
    return out


def resident_mask(w: Workload, layer: int) -> np.ndarray:
    """uint8 [E]: 1 = expert resident in this layer's table row."""
    mask = np.empty(w.n_experts, dtype=np.uint8)
    perm = np.empty(w.n_experts, dtype=np.int32)
    n_res = w.n_experts if w.n_resident < 0 else w.n_resident
    lib().synth_resident_mask(w.seed, layer, w.n_experts, n_res, mask.ctypes.data, perm.ctypes.data)
    return mask


def permutation(tag: int, a: int, n: int, seed: int = 0) -> np.ndarray:
    perm = np.empty(n, dtype=np.int32)
    lib().synth_permutation(seed, tag, a, n, perm.ctypes.data)
    return perm
