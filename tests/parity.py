"""Helpers shared by the GPU parity tests: run the oracle and the CUDA path on
the same seeded workload and compare."""
import numpy as np
import torch

import oracle as O
import workloads as W


def np_elems(t, dtype):
    """CPU tensor -> numpy array the oracle takes (fp32, or raw bf16 bits)."""
    t = t.detach().cpu().contiguous()
    return t.numpy() if dtype == W.F32 else t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(a):
    return (a.astype(np.uint32) << 16).view(np.float32)


def out_as_f32(t, dtype):
    t = t.detach().cpu().contiguous()
    return t.numpy() if dtype == W.F32 else t.float().numpy()


def oracle_mask(w):
    return O.mask_build(w.parent.numpy(), w.tree_off.numpy(), w.n_max)


def oracle_attention(w, rows=None):
    return O.tree_attention(np_elems(w.q, w.dtype), np_elems(w.k_cache, w.dtype), np_elems(w.v_cache, w.dtype),
                            w.block_table.numpy(), w.block_size, w.prefix_len.numpy(), w.tree_off.numpy(),
                            w.parent.numpy(), w.n_max, w.Hq, w.Hkv, w.D, w.dtype, w.scale, rows=rows)


def oracle_greedy(w):
    return O.verify_greedy(w.p_logits.numpy(), w.tokens.numpy(), w.parent.numpy(), w.tree_off.numpy(), w.n_max)


def oracle_stochastic(w):
    return O.verify_stochastic(w.p_logits.numpy(), w.q_probs.numpy(), w.tokens.numpy(), w.parent.numpy(),
                               w.tree_off.numpy(), w.uniforms.numpy().view(np.uint32), w.n_max)


def attn_tolerance_ok(got, ref, dtype):
    """fp32: max-abs 1e-5.  bf16 inputs: |got - ref| <= 2e-2 + 1e-2 |ref|."""
    if dtype == W.F32:
        return np.abs(got - ref) <= 1e-5
    return np.abs(got - ref) <= 2e-2 + 1e-2 * np.abs(ref)
