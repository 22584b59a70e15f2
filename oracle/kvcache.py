"""Reference model of the multi-shot NVFP4 KV cache's frame policy -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this module; it shares nothing with the product (the C++ cache manager
and the CUDA gather-dequant).

What it models ("LongLive-2.0: An NVFP4 Parallel Infrastructure for Long Video
Generation", summary page):
  - inference step 7: the KV cache is written one chunk of F_c latent frames at a
    time (K smoothed, then NVFP4 with 4/6 block scales);
  - inference step 9: attention over a Global Sink (the first S_g frames of the
    video) plus a Shot-Level Sink (the first S_s frames of the current shot, held
    as START/LEN pointers into frames that are already cached, so it costs no
    memory of its own); a prompt switch rebinds the shot sink.
Readings where the page is silent (each also listed with the design notes):
  - K1 the local part of the attention is a rolling window of the W frames right
    before the chunk being generated (the cache-read workload: 3 sink frames + 18
    rolling frames);
  - K2 a prompt switch happens between chunks: the next chunk is the new shot's
    first, START = its first frame, and LEN = min(S_s, frames of the shot cached so far);
  - K3 the view is the set union of the three ranges in ascending frame order (a
    frame that is both sink and window appears once);
  - K4 a frame can be dropped once no later view can contain it: after chunk n is
    written the next view is chunk n + 1's, windows only move forward and a new
    shot sink only covers frames not yet written.
"""
from __future__ import annotations


def view_frames(n_chunks: int, frames_per_chunk: int, global_sink: int, shot_sink: int, window: int,
                shot_start: int) -> list[int]:
    """Frames (video frame indices) that chunk ``n_chunks`` attends to, ascending (K1-K3).

    ``n_chunks`` chunks are cached, so frames [0, n_chunks * frames_per_chunk) exist."""
    cur = n_chunks * frames_per_chunk
    out = []
    for f in range(cur):
        in_global = f < global_sink
        in_shot = shot_start <= f < shot_start + shot_sink
        in_window = f >= cur - window
        if in_global or in_shot or in_window:
            out.append(f)
    return out


class CacheModel:
    """The cache as a sequence of events: append a chunk, switch the prompt, read a view.

    Keeps which chunks are resident; a chunk is released (K4) when none of its frames
    can be in the next chunk's view or a later one."""

    def __init__(self, frames_per_chunk: int, global_sink: int, shot_sink: int, window: int):
        self.F = frames_per_chunk
        self.S_g, self.S_s, self.W = global_sink, shot_sink, window
        self.n_chunks = 0
        self.shot_start = 0
        self.resident: set[int] = set()

    def view(self) -> list[int]:
        return view_frames(self.n_chunks, self.F, self.S_g, self.S_s, self.W, self.shot_start)

    def _needed_after_append(self, chunk: int) -> bool:
        # frames the view of chunk (n_chunks + 1) can hold, once chunk n_chunks is written
        nxt = (self.n_chunks + 1) * self.F
        for f in range(chunk * self.F, (chunk + 1) * self.F):
            if f < self.S_g or self.shot_start <= f < self.shot_start + self.S_s or f >= nxt - self.W:
                return True
        return False

    def append(self) -> int:
        """Writes chunk n_chunks; returns its index. Releases dead chunks first."""
        self.resident = {c for c in self.resident if self._needed_after_append(c)}
        c = self.n_chunks
        self.resident.add(c)
        self.n_chunks += 1
        return c

    def new_shot(self) -> None:
        """Prompt switch: the next chunk is the first of a new shot."""
        self.shot_start = self.n_chunks * self.F
