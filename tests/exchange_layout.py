"""A plain restatement of the head-shard segment layout (include/nvfp4.h, "Head shards of
a quantized KV tensor"), used by the exchange tests to build and read segments on the CPU."""
import numpy as np


def pad16(n: int) -> int:
    return (n + 15) // 16 * 16


def seg_bytes(T, H, D, P, with_mean):
    hs = H // P
    return 16 + (hs * D * 4 if with_mean else 0) + pad16(T * hs * D // 2) + pad16(T * hs * D // 16)


def pack(codes, scales, g, mean, P):
    """codes [T][H][D/2], scales [T][H][D/16], g float, mean [H][D] or None -> uint8 [P][seg]."""
    T, H, D2 = codes.shape
    D = 2 * D2
    hs = H // P
    out = np.zeros((P, seg_bytes(T, H, D, P, mean is not None)), np.uint8)
    for p in range(P):
        b = out[p]
        b[0:4] = np.array([g], np.float32).view(np.uint8)
        o = 16
        if mean is not None:
            m = np.ascontiguousarray(mean.reshape(H, D)[p * hs:(p + 1) * hs], np.float32).view(np.uint8).ravel()
            b[o:o + m.size] = m
            o += m.size
        c = np.ascontiguousarray(codes[:, p * hs:(p + 1) * hs]).ravel()
        b[o:o + c.size] = c
        o += pad16(c.size)
        s = np.ascontiguousarray(scales[:, p * hs:(p + 1) * hs]).ravel()
        b[o:o + s.size] = s
    return out


def unpack(segs, T, H, D, P, with_mean):
    """uint8 [P][seg] (row r from rank r) -> codes [P T][H/P][D/2], scales, g [P], means [P][H/P][D] or None."""
    hs = H // P
    codes = np.zeros((P * T, hs, D // 2), np.uint8)
    scales = np.zeros((P * T, hs, D // 16), np.uint8)
    gs = np.zeros(P, np.float32)
    means = np.zeros((P, hs, D), np.float32) if with_mean else None
    for r in range(P):
        b = segs[r]
        gs[r] = b[0:4].view(np.float32)[0]
        o = 16
        if with_mean:
            n = hs * D * 4
            means[r] = b[o:o + n].view(np.float32).reshape(hs, D)
            o += n
        n = T * hs * D // 2
        codes[r * T:(r + 1) * T] = b[o:o + n].reshape(T, hs, D // 2)
        o += pad16(n)
        n = T * hs * D // 16
        scales[r * T:(r + 1) * T] = b[o:o + n].reshape(T, hs, D // 16)
    return codes, scales, gs, means
