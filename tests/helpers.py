"""Helpers shared by the tests (not by the product or the oracle)."""
import numpy as np


def bf16_exact(a):
    """bf16 bit patterns (uint16) of values that are exactly representable in bf16."""
    a = np.asarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def bf16_to_f64(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_rne_np(x):
    """Round fp64 values to the nearest bf16 (ties to even) with numpy, written
    independently of the oracle: x = m * 2^e, keep 8 significant bits."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    q = np.maximum(e - 8, -133)
    y = np.ldexp(np.rint(np.ldexp(x, -q)), q)
    return bf16_exact(y.astype(np.float32))


def permutation(n, seed):
    return np.random.default_rng(seed).permutation(n)


def perm_matrix(rows, cols, src):
    """M[i, src[i]] = 1: (M x)[i] = x[src[i]]."""
    m = np.zeros((rows, cols), np.float32)
    m[np.arange(rows), src] = 1.0
    return m
