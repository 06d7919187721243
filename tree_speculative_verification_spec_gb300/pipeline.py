"""One verification pass through the C ABI: buffers + the five calls in order.

VerifyPass owns the device outputs and workspaces of one batch shape and
enqueues, on one stream and with no host synchronisation:
  spec_tree_mask_build -> [spec_kv_append] -> spec_tree_attention ->
  spec_tree_verify_{greedy, stochastic} -> spec_kv_commit.
Allocation happens once, in the constructor; run() only launches.
"""
from dataclasses import dataclass

import torch

from . import _binding as S


@dataclass
class DeviceBatch:
    """Device-resident inputs of one pass (all CUDA tensors)."""
    B: int
    T: int
    n_max: int
    V: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    max_prefix: int
    parent: torch.Tensor
    tree_off: torch.Tensor
    tokens: torch.Tensor
    prefix_len: torch.Tensor
    block_table: torch.Tensor
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    p_logits: torch.Tensor
    q_probs: torch.Tensor
    uniforms: torch.Tensor  # int32 [T, 2] raw words
    scale: float

    @property
    def max_blocks(self):
        return self.block_table.shape[1]

    @classmethod
    def from_workload(cls, w, device="cuda", max_prefix=None):
        def d(t):
            return None if t is None else t.to(device, non_blocking=False).contiguous()
        mp = int(w.prefix_len.max()) if max_prefix is None and w.B > 0 else (max_prefix or 0)
        return cls(B=w.B, T=w.T, n_max=w.n_max, V=w.V, Hq=w.Hq, Hkv=w.Hkv, D=w.D, block_size=w.block_size,
                   num_blocks=w.num_blocks, max_prefix=mp, parent=d(w.parent), tree_off=d(w.tree_off),
                   tokens=d(w.tokens), prefix_len=d(w.prefix_len), block_table=d(w.block_table), q=d(w.q),
                   k_cache=d(w.k_cache), v_cache=d(w.v_cache), p_logits=d(w.p_logits), q_probs=d(w.q_probs),
                   uniforms=d(w.uniforms), scale=w.scale)


class VerifyPass:
    # stochastic verification options used when verify() is not given them:
    # per-request inverse temperatures (float32 device tensor [B], or None for
    # 1) and the draft-row layout
    inv_temp = None
    q_layout = S.SPEC_Q_PER_PARENT

    def __init__(self, batch: DeviceBatch):
        b = batch
        dev = b.q.device
        i32 = dict(dtype=torch.int32, device=dev)
        self.W = (b.n_max + 63) // 64
        self.mask = torch.zeros((max(b.T, 1), self.W), dtype=torch.int64, device=dev)
        self.depth = torch.zeros(max(b.T, 1), **i32)
        self.status = torch.zeros(max(b.B, 1), **i32)
        self.out = torch.empty_like(b.q)
        aws = S.spec_attention_workspace_size(b.B, b.T, b.n_max, b.max_prefix, b.Hq, b.Hkv, b.D)
        self.attn_ws = torch.empty(aws, dtype=torch.uint8, device=dev)
        vws = S.spec_verify_workspace_size(b.B, b.n_max, b.V)
        self.verify_ws = torch.empty(vws, dtype=torch.uint8, device=dev)
        self.path = torch.full((max(b.B, 1), b.n_max), -1, **i32)
        self.accept_len = torch.zeros(max(b.B, 1), **i32)
        self.emitted = torch.full((max(b.B, 1), b.n_max), -1, **i32)
        self.n_emitted = torch.zeros(max(b.B, 1), **i32)
        self.new_len = torch.zeros(max(b.B, 1), **i32)
        self.batch = b

    def mask_build(self, stream=None):
        b = self.batch
        S.spec_tree_mask_build(b.parent, b.tree_off, b.B, b.n_max, self.mask, self.depth, self.status, stream)

    def append(self, k_new, v_new, stream=None):
        """Tree K/V rows [T][Hkv][D] into slots prefix_len + u (before attention)."""
        b = self.batch
        S.spec_kv_append(k_new, v_new, b.k_cache, b.v_cache, b.block_table, b.max_blocks, b.block_size,
                         b.num_blocks, b.prefix_len, b.tree_off, b.B, b.n_max, b.Hkv, b.D, self.status, stream)

    def attention(self, flags=S.SPEC_ATTN_AUTO, stream=None):
        b = self.batch
        S.spec_tree_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.max_blocks, b.block_size, b.num_blocks,
                              b.prefix_len, b.tree_off, self.mask, b.B, b.T, b.n_max, b.max_prefix, b.Hq, b.Hkv, b.D,
                              b.scale, self.out, self.attn_ws, self.status, flags, stream)

    def verify(self, mode="stochastic", stream=None, inv_temp=None, q_layout=None):
        b = self.batch
        inv_temp = self.inv_temp if inv_temp is None else inv_temp
        q_layout = self.q_layout if q_layout is None else q_layout
        if mode == "greedy":
            S.spec_tree_verify_greedy(b.p_logits, b.tokens, b.parent, b.tree_off, b.B, b.n_max, b.V, self.path, self.accept_len, self.emitted, self.n_emitted,
                                      self.verify_ws, self.status, stream)
        else:
            S.spec_tree_verify_stochastic(b.p_logits, b.q_probs, b.tokens, b.parent, b.tree_off, b.uniforms, b.B,
                                          b.n_max, b.V, self.path, self.accept_len, self.emitted, self.n_emitted,
                                          self.verify_ws, self.status, stream, inv_temp=inv_temp, q_layout=q_layout)

    def commit(self, stream=None):
        b = self.batch
        S.spec_kv_commit(b.k_cache, b.v_cache, b.block_table, b.max_blocks, b.block_size, b.num_blocks,
                         b.prefix_len, self.path, b.n_max, self.accept_len, b.B, b.Hkv, b.D, self.new_len,
                         self.status, stream)

    def run(self, mode="stochastic", attn_flags=S.SPEC_ATTN_AUTO, commit=True, stream=None, tree_kv=None):
        """tree_kv: (k_new, v_new) rows appended before attention, or None when
        the tree K/V are already in the cache."""
        self.mask_build(stream)
        if tree_kv is not None:
            self.append(*tree_kv, stream=stream)
        self.attention(attn_flags, stream)
        self.verify(mode, stream)
        if commit:
            self.commit(stream)
