"""ctypes binding of the measurement library ``libta11_probe.so`` (csrc/probe.h).

Roof microbenchmarks for the benchmark's tables: the special-function unit's exp2
rate and the tensor core's rate for the score GEMM's UMMA shape.  Not part of the
attention library's interface; nothing on the attention path loads it.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libta11_probe.so")
EXPORTED = ("ta11_probe_ex2", "ta11_probe_umma", "ta11_probe_status")

_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"measurement library not built: {LIB_PATH} is missing")
    L = ctypes.CDLL(LIB_PATH)
    vp, i = ctypes.c_void_p, ctypes.c_int
    L.ta11_probe_ex2.argtypes = [vp, i, i, vp]
    L.ta11_probe_ex2.restype = i
    L.ta11_probe_umma.argtypes = [i, i, ctypes.c_ulonglong, vp]
    L.ta11_probe_umma.restype = i
    L.ta11_probe_status.argtypes = [i]
    L.ta11_probe_status.restype = i
    _lib = L
    return L


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise RuntimeError(f"{where}: status {rc}")


def _time(run, stream, reps: int) -> float:
    """Median milliseconds of `run` over `reps` CUDA-event timings after one warm-up."""
    run()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    ts.sort()
    return ts[len(ts) // 2]


def ex2_rate(device=None, iters: int = 2048, reps: int = 5) -> float:
    """exp2 per second of the special-function units (4 blocks of 512 threads per SM)."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    n_blocks = 4 * torch.cuda.get_device_properties(dev).multi_processor_count
    out = torch.empty(n_blocks * 512, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ms = _time(lambda: _check(lib().ta11_probe_ex2(out.data_ptr(), n_blocks, iters, stream.cuda_stream),
                              "ta11_probe_ex2"), stream, reps)
    return n_blocks * 512 * 8 * iters / (ms * 1e-3)


def ex2_values(n_blocks: int, iters: int, device=None) -> torch.Tensor:
    """Each thread's sum of its 8 exp2 chains after `iters` steps (n_blocks * 512 floats)."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    out = torch.empty(n_blocks * 512, dtype=torch.float32, device=dev)
    _check(lib().ta11_probe_ex2(out.data_ptr(), n_blocks, iters, torch.cuda.current_stream(dev).cuda_stream),
           "ta11_probe_ex2")
    return out


def umma_rate(device=None, iters: int = 1024, reps: int = 5, limit_ns: int = 2_000_000_000) -> float:
    """bf16 FLOP/s of the tensor cores for the score GEMM's UMMA shape (one CTA per SM)."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    n = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = torch.cuda.current_stream(dev)
    ms = _time(lambda: _check(lib().ta11_probe_umma(n, iters, limit_ns, stream.cuda_stream), "ta11_probe_umma"),
               stream, reps)
    return n * iters * 8 * 2.0 * 128 * 128 * 16 / (ms * 1e-3)


def status(reset: bool = False) -> int:
    """The probes' status word (synchronises the device first): 0, or 7 after a timeout."""
    torch.cuda.synchronize()
    return lib().ta11_probe_status(int(bool(reset)))
