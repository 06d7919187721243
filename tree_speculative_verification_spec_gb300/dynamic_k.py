"""Dynamic draft length around the verification pass ("Hardware-aware dynamic
speculative decoding"): a goodput table kept by the library's host functions,
and full CUDA graphs of the pass, one per <tokens, K>.

The arithmetic of the policy (argmax of AL / ITL, the lookup, the moving
average, the graph keys) is in the library (csrc/dsd.cu); this module holds
the tables and the captured graphs.
"""
import numpy as np
import torch

from . import _binding as S


class DynamicK:
    """Per profiled batch size and draft length: acceptance length (AL) and
    inter-token latency (ITL); the K of highest goodput = AL / ITL per batch
    size; the K for the batch size of a step.  Cells start unmeasured (NaN)."""

    def __init__(self, bs_values, k_values):
        self.bs_values = np.ascontiguousarray(bs_values, dtype=np.int32)
        self.k_values = np.ascontiguousarray(k_values, dtype=np.int32)
        shape = (len(self.bs_values), len(self.k_values))
        self.al = np.full(shape, np.nan)
        self.itl = np.full(shape, np.nan)

    def record(self, bs_index, k_index, al, itl, weight=1.0):
        """Folds a measurement into a cell (weight 1: replace; below 1: moving average)."""
        S.spec_dsd_update(self.al, self.itl, bs_index, k_index, float(al), float(itl), float(weight))

    def optimal_k(self):
        out = np.zeros(len(self.bs_values), np.int32)
        S.spec_dsd_optimal_k(self.al, self.itl, self.k_values, out)
        return out

    def select(self, bs):
        """The K for batch size `bs`, from the rows that have a measurement."""
        k_opt = self.optimal_k()
        ok = k_opt >= 0
        if not ok.any():
            raise ValueError("no measured row in the goodput table")
        return S.spec_dsd_select_k(np.ascontiguousarray(self.bs_values[ok]), np.ascontiguousarray(k_opt[ok]), bs)


class GraphCache:
    """Full CUDA graphs of one verification pass per <tokens, K> ("Compatibility
    with full CUDA Graph"): `make_pass(tokens, K)` returns a VerifyPass over
    static buffers; its first use runs the pass once, captures it, and later
    uses replay the graph.  New inputs are copied into the pass's buffers
    before a replay."""

    def __init__(self, make_pass, mode="stochastic", attn_flags=0, commit=True):
        self._make = make_pass
        self._mode, self._flags, self._commit = mode, attn_flags, commit
        self._entries = {}

    def keys(self):
        return sorted(self._entries)

    def pass_for(self, tokens, K):
        return self._entry(tokens, K)[1]

    def _entry(self, tokens, K):
        key = (int(tokens), int(K))
        if key not in self._entries:
            vp = self._make(*key)
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                vp.run(self._mode, self._flags, self._commit)  # first calls set kernel attributes
            torch.cuda.current_stream().wait_stream(side)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                vp.run(self._mode, self._flags, self._commit)
            self._entries[key] = (g, vp)
        return self._entries[key]

    def replay(self, tokens, K):
        g, vp = self._entry(tokens, K)
        g.replay()
        return vp
