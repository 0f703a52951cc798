"""Compile tests/host/mask_host.cpp (host-only build of the kernels' mask rules)."""
import ctypes
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
SRC = os.path.join(HERE, "mask_host.cpp")
OUT = os.path.join(HERE, "_mask_host.so")
DEPS = [SRC, os.path.join(ROOT, "exact_io_aware_13_gb300", "csrc", "mask.cuh"),
        os.path.join(ROOT, "include", "attn.h")]


def load() -> ctypes.CDLL:
    if not os.path.exists(OUT) or os.path.getmtime(OUT) < max(map(os.path.getmtime, DEPS)):
        tmp = OUT + f".{os.getpid()}.tmp"
        subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-x", "c++", SRC,
                        "-I", os.path.join(ROOT, "include"),
                        "-I", os.path.join(ROOT, "exact_io_aware_13_gb300", "csrc"),
                        "-o", tmp], check=True)
        os.replace(tmp, OUT)
    return ctypes.CDLL(OUT)
