"""Seeded synthetic inputs for the VSA forward (shared by tests, smoke and bench).

This module draws random numbers and lays them out; it holds none of the
attention method's arithmetic. Both the CUDA path and the CPU oracle receive
the exact bf16 bytes it returns.

Recipe (stands in for the FastH3 request shapes of "UniServe: serving FastH3 at
its fastest", section "The FastH3 workload": 56 heads x 128, 72,576 video
tokens for a 10 s request; no checkpoint or dataset is used):

* Q, K, V, gate are ``[B, N, H, 128]`` token-major, segments in memory order
  text | audio | video, N = len_text + len_audio + len_video.
* Q, K, V ~ N(0, 1) i.i.d.; gate pre-activation ~ N(0, 1).
* For every (batch, head, 64-token video tile) one offset vector ~ N(0, 0.5^2)
  is added to both Q and K on that tile's video tokens (prefix rows are not
  shifted). This gives each query tile a strongly preferred key tile, the
  locality structure a video's block-sparse pattern has.
* Draw order: Q, K, V, offsets, gate, from one ``torch.Generator`` seeded with
  the config's seed, in fp32 on ``device``; then rounded to bf16 (RNE).

Values depend on the device the generator runs on (torch's CPU and CUDA
generators are different streams); every test hands the same tensors to both
sides, so that does not matter for parity.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

TILE = 64
HEAD_DIM = 128


@dataclass(frozen=True)
class Config:
    name: str
    batch: int
    heads: int
    len_text: int
    len_audio: int
    len_video: int
    keep: tuple = (0.2,)
    seed: int = 0
    head_dim: int = HEAD_DIM

    @property
    def prefix(self) -> int:
        return self.len_text + self.len_audio

    @property
    def seq(self) -> int:
        return self.prefix + self.len_video

    @property
    def n_video_tiles(self) -> int:
        return -(-self.len_video // TILE)


# The five workloads: tiny oracle case, medium, one GPU's head share of a 5 s
# request, the full 10 s FastH3 shape on one GPU, and a ragged sparsity sweep.
CONFIGS = {
    "tiny": Config("tiny", 1, 2, 64, 64, 1024, (0.2,), 0),
    "medium": Config("medium", 1, 14, 1024, 512, 8192, (0.2,), 1),
    "5s": Config("5s", 1, 14, 1024, 1024, 36288, (0.2,), 2),
    "10s": Config("10s", 1, 56, 1024, 1024, 72576, (0.2,), 3),
    "ragged": Config("ragged", 2, 56, 1000, 700, 72500, (0.1, 0.2, 0.4), 4),
}


def make_inputs(batch, heads, len_text, len_audio, len_video, seed, device="cpu",
                head_dim=HEAD_DIM, offset_std=0.5):
    """Return (q, k, v, gate) bf16 tensors of shape [B, N, H, head_dim] on ``device``."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    prefix = len_text + len_audio
    n = prefix + len_video
    shape = (batch, n, heads, head_dim)
    q = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    k = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    n_tiles = -(-len_video // TILE)
    off = torch.randn((batch, n_tiles, heads, head_dim), generator=gen, device=device,
                      dtype=torch.float32) * offset_std
    full = len_video // TILE
    if full:
        body = slice(prefix, prefix + full * TILE)
        shift = off[:, :full].unsqueeze(2)  # [B, full, 1, H, D]
        for x in (q, k):
            x[:, body].view(batch, full, TILE, heads, head_dim).add_(shift)
    if full < n_tiles:  # ragged last tile
        tail = slice(prefix + full * TILE, n)
        for x in (q, k):
            x[:, tail].add_(off[:, full].unsqueeze(1))
    gate = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    out = []
    for x in (q, k, v, gate):
        out.append(x.to(torch.bfloat16))
    del q, k, v, gate
    return tuple(out)


def make_config_inputs(cfg: Config, device="cpu"):
    return make_inputs(cfg.batch, cfg.heads, cfg.len_text, cfg.len_audio, cfg.len_video,
                       cfg.seed, device=device, head_dim=cfg.head_dim)


def bf16_bits(t: torch.Tensor):
    """The raw bf16 bit patterns of a CPU tensor as a numpy uint16 array (no conversion)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view("uint16")


# ---------------------------------------------------------------- preprocessing inputs
#
# Recipe for the fused-preprocessing inputs (the projections before Q/K norm and
# RoPE, as "Fused attention preprocessing" receives them):
# * one merged bf16 projection buffer [B, rows_in, 4, H, 128] (Q, K, V, gate
#   side by side in each row, as one merged projection writes them), values
#   N(0, 1) times a per-(row, tensor, head) scale exp(N(0, 0.5^2)), so rows
#   differ in RMS. rows_in is a capacity that may exceed the token count;
# * RMSNorm weights 1 + N(0, 0.1^2), fp32 [H, 128], one set for Q and one for K;
# * RoPE tables for 3-D positions: video token v sits at (frame, y, x) of a
#   24 x 42 latent grid per frame (1,008 tokens a frame: 72 frames are the
#   72,576 tokens of a 10 s request at 1344 x 768). Text and audio token n sit
#   at (n, 0, 0). The rope_dim / 2 angles split evenly over the three axes,
#   with frequencies 10000^(-j / per_axis);
# * a row map: a random injective choice of projection rows for the tokens.

FRAME_GRID = (24, 42)


def make_projections(batch, rows_in, heads, seed, device="cpu", head_dim=HEAD_DIM):
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    x = torch.randn((batch, rows_in, 4, heads, head_dim), generator=gen, device=device, dtype=torch.float32)
    scale = torch.exp(0.5 * torch.randn((batch, rows_in, 4, heads, 1), generator=gen, device=device,
                                        dtype=torch.float32))
    return (x * scale).to(torch.bfloat16)


def make_norm_weights(heads, seed, head_dim=HEAD_DIM):
    gen = torch.Generator()
    gen.manual_seed(int(seed))
    w = 1.0 + 0.1 * torch.randn((2, heads, head_dim), generator=gen, dtype=torch.float32)
    return w[0].contiguous(), w[1].contiguous()


def rope_positions(len_text, len_audio, len_video):
    """int64 [N, 3] (frame, y, x) position of each token, segments text | audio | video."""
    prefix = len_text + len_audio
    pos = torch.zeros((prefix + len_video, 3), dtype=torch.int64)
    pos[:prefix, 0] = torch.arange(prefix)
    v = torch.arange(len_video)
    per_frame = FRAME_GRID[0] * FRAME_GRID[1]
    pos[prefix:, 0] = v // per_frame
    pos[prefix:, 1] = (v % per_frame) // FRAME_GRID[1]
    pos[prefix:, 2] = v % FRAME_GRID[1]
    return pos


def make_rope_tables(len_text, len_audio, len_video, rope_dim):
    """fp32 (cos, sin), each [N, rope_dim / 2], for the 3-D positions above."""
    half = rope_dim // 2
    pos = rope_positions(len_text, len_audio, len_video).to(torch.float64)
    per_axis = [half // 3 + (1 if a < half % 3 else 0) for a in range(3)]
    angles = []
    for axis, m in enumerate(per_axis):
        freq = 10000.0 ** (-torch.arange(m, dtype=torch.float64) / max(m, 1))
        angles.append(pos[:, axis:axis + 1] * freq[None])
    th = torch.cat(angles, dim=1) if half else torch.zeros((pos.shape[0], 0), dtype=torch.float64)
    return torch.cos(th).to(torch.float32).contiguous(), torch.sin(th).to(torch.float32).contiguous()


def make_row_map(batch, n_tokens, rows_in, seed):
    """int32 [B, N]: distinct projection rows, a random choice per batch."""
    gen = torch.Generator()
    gen.manual_seed(int(seed))
    return torch.stack([torch.randperm(rows_in, generator=gen)[:n_tokens] for _ in range(batch)]).to(torch.int32)
