"""Places a generated workload in device memory and drives the library on it.

Used by the GPU tests, the smoke check and the benchmark.  It moves bytes and
calls the C ABI (through the package's binding); it computes nothing itself.
"""

from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_arena_gb300 as K

# 0x7FC1 is a NaN in both binary16 and bfloat16: any read of an unused arena
# slot that reaches an output poisons it.
NAN_SENTINEL = 0x7FC1


def _dt(w):
    return torch.float16 if w.dtype == "f16" else torch.bfloat16


def to_device_bits(a: np.ndarray, dtype, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(dtype)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceWorkload:
    """Device copies of one workload: step inputs, arena, tables, workspace."""

    def __init__(self, w, device: str = "cuda", sentinel: int = NAN_SENTINEL, fill_prefix: bool = True):
        self.w = w
        self.device = device
        dt = _dt(w)
        self.dtype = dt
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
        self.q = to_device_bits(w.q, dt, device)
        k_new, v_new = w.step_kv()
        self.k_new = to_device_bits(k_new, dt, device)
        self.v_new = to_device_bits(v_new, dt, device)
        self.q_rot = torch.empty_like(self.q)
        shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
        s16 = np.array([sentinel], dtype=np.uint16).view(np.int16)[0]
        self.k_arena = torch.full(shape, int(s16), dtype=torch.int16, device=device).view(dt)
        self.v_arena = torch.full(shape, int(s16), dtype=torch.int16, device=device).view(dt)
        self.block_tables = i32(w.block_tables)
        self.context_lens = i32(w.context_lens)
        self.query_start_loc = i32(w.query_start_loc)
        self.positions = i32(w.positions)
        self.rope_max_pos = max(w.max_context_len, 1)
        self.rope_table = torch.from_numpy(K.kshipra_rope_table_build(self.rope_max_pos, w.head_dim, w.theta)).to(device)
        self.out = torch.empty_like(self.q)
        self.ws_bytes = K.kshipra_paged_attention_workspace_size(w.num_seqs, w.num_tokens, w.max_context_len,
                                                                 w.num_q_heads, w.num_kv_heads, w.head_dim)
        self.workspace = torch.empty(max(self.ws_bytes, 1), dtype=torch.uint8, device=device)
        if fill_prefix:
            self.append_prefix()

    def append_prefix(self, stream=None):
        kp, vp, qsl_p, pos_p = self.w.prefix_batch()
        if len(pos_p) == 0:
            return
        kd = to_device_bits(kp, self.dtype, self.device)
        vd = to_device_bits(vp, self.dtype, self.device)
        qsl = torch.from_numpy(qsl_p).to(self.device)
        pos = torch.from_numpy(pos_p).to(self.device)
        K.kshipra_kv_append_rope(None, kd, vd, None, self.k_arena, self.v_arena, self.block_tables, qsl, pos,
                                 self.rope_table, stream=stream)

    def append_step(self, stream=None):
        K.kshipra_kv_append_rope(self.q, self.k_new, self.v_new, self.q_rot, self.k_arena, self.v_arena,
                                 self.block_tables, self.query_start_loc, self.positions, self.rope_table,
                                 stream=stream)

    def attention(self, out=None, stream=None):
        w = self.w
        K.kshipra_paged_attention(self.out if out is None else out, self.q_rot, self.k_arena, self.v_arena,
                                  self.block_tables, self.context_lens, self.query_start_loc, self.positions,
                                  w.max_query_len, w.max_context_len, w.scale, self.workspace, stream=stream)

    def step(self, stream=None):
        self.append_step(stream)
        self.attention(stream=stream)

    def decode_step(self, q_rot=True, stream=None):
        """Append and attention through kshipra_decode_step (one launch for
        decode-class batches); q_rot=False passes no q_rot buffer."""
        w = self.w
        K.kshipra_decode_step(self.out, self.q, self.k_new, self.v_new, self.q_rot if q_rot else None, self.k_arena,
                              self.v_arena, self.block_tables, self.context_lens, self.query_start_loc,
                              self.positions, self.rope_table, w.max_query_len, w.max_context_len, w.scale,
                              self.workspace, stream=stream)

    def out_f64(self) -> np.ndarray:
        return self.out.float().cpu().numpy().astype(np.float64)
