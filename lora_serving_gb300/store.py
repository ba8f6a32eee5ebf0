"""Device-resident adapter store and batch metadata (memory management only).

The store layout is the one the kernels read (peft orientation, K-major):
  A: bf16 [n_slots][r_slot][h_in]      per projection
  B: bf16 [n_slots][width][r_slot]     per projection, scale already folded
Slots are ``max_loras`` GPU slots and ``r_slot`` the slot rank
(``max_lora_rank``) of the vLLM offline LoRA page, step 2.  Folding and
padding happen in the C library (``lora_prepare_adapter``); this module only
allocates torch tensors, fills host staging buffers through the C call and
copies them to the device.
"""
from __future__ import annotations

import numpy as np
import torch

from . import abi


def _bits_to_device(a: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return t.to(device, non_blocking=False)


class GroupStore:
    """Adapter store of one projection group (projections sharing x)."""

    def __init__(self, h_in: int, projs, n_slots: int, r_slot: int, device="cuda"):
        self.h_in, self.n_slots, self.r_slot = int(h_in), int(n_slots), int(r_slot)
        self.projs = [(str(n), int(w)) for n, w in projs]
        self.offsets = []
        o = 0
        for _, w in self.projs:
            self.offsets.append(o)
            o += w
        self.ld_y = o
        self.device = device
        self.A = [torch.zeros(n_slots, r_slot, h_in, dtype=torch.bfloat16, device=device) for _ in self.projs]
        self.B = [torch.zeros(n_slots, w, r_slot, dtype=torch.bfloat16, device=device) for _, w in self.projs]
        self._c = None

    def load_slots(self, adapters):
        """adapters: {slot: [(A_bits [r][h_in], B_bits [w][r], alpha, use_rslora) per projection]}."""
        for p, (_, w) in enumerate(self.projs):
            hA = np.zeros((self.n_slots, self.r_slot, self.h_in), np.uint16)
            hB = np.zeros((self.n_slots, w, self.r_slot), np.uint16)
            touched = []
            for k, per_proj in adapters.items():
                A, B, alpha, rs = per_proj[p]
                abi.lora_prepare_adapter(A, B, alpha, rs, self.r_slot, hA[k], hB[k])
                touched.append(k)
            if not touched:
                continue
            if len(touched) == self.n_slots:
                self.A[p].copy_(_bits_to_device(hA, "cpu"))
                self.B[p].copy_(_bits_to_device(hB, "cpu"))
            else:
                for k in touched:
                    self.A[p][k].copy_(_bits_to_device(hA[k], "cpu"))
                    self.B[p][k].copy_(_bits_to_device(hB[k], "cpu"))
        self._c = None
        return self

    @classmethod
    def from_workload(cls, wl, group_name: str, device="cuda"):
        g = next(g for g in wl.groups if g.name == group_name)
        st = cls(g.h_in, g.projs, wl.n_slots, wl.r_slot, device)
        adapters = {}
        for k in range(wl.n_slots):
            adapters[k] = [(wl.A[(g.name, pn, k)], wl.B[(g.name, pn, k)], float(wl.alphas[k]),
                            bool(wl.rslora[k])) for pn, _ in g.projs]
        return st.load_slots(adapters)

    def c_projs(self):
        """ctypes lora_proj_t array (kept alive by this object)."""
        if self._c is None:
            self._c = abi.make_projs([(self.A[p], self.B[p], self.offsets[p], w)
                                      for p, (_, w) in enumerate(self.projs)])
        return self._c

    def nbytes_slot(self) -> int:
        """Bytes of one slot across the group's projections."""
        return sum(self.r_slot * (self.h_in + w) * 2 for _, w in self.projs)


class BatchMeta:
    """Batch metadata from the C builder, copied to the device."""

    def __init__(self, ids, n_prefill: int, n_slots: int, device="cuda"):
        ids = np.ascontiguousarray(ids, np.int32)
        m = abi.lora_build_metadata(ids, n_prefill, n_slots)
        self.host = m
        self.host_ids = ids

        def up(a):
            a = np.ascontiguousarray(a, np.int32)
            if a.size == 0:
                a = np.zeros(1, np.int32)
            return torch.from_numpy(a).to(device)

        self.ids = up(ids)
        self.seg_starts = up(m["seg_starts"])
        self.seg_slot = up(m["seg_slot"])
        self.perm = up(m["perm"])
        self.gseg_starts = up(m["gseg_starts"])
        self.gseg_slot = up(m["gseg_slot"])
        self.n_rows, self.n_prefill = int(ids.size), int(n_prefill)
        c = abi.lora_meta_t()
        c.lora_ids = self.ids.data_ptr()
        c.n_rows, c.n_prefill = self.n_rows, self.n_prefill
        c.seg_starts, c.seg_slot = self.seg_starts.data_ptr(), self.seg_slot.data_ptr()
        c.n_segs, c.max_seg_len = m["n_segs"], m["max_seg_len"]
        c.perm, c.gseg_starts, c.gseg_slot = (self.perm.data_ptr(), self.gseg_starts.data_ptr(),
                                              self.gseg_slot.data_ptr())
        c.n_gsegs, c.max_gseg_len = m["n_gsegs"], m["max_gseg_len"]
        self.c = c


def workspace_for(n_rows: int, n_proj: int, r_slot: int, device="cuda") -> torch.Tensor:
    nbytes = max(abi.lora_apply_workspace_bytes(n_rows, n_proj, r_slot), 256)
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def apply(y: torch.Tensor, x: torch.Tensor, store: GroupStore, meta: BatchMeta,
          workspace: torch.Tensor, dev_status=None, stream=None, flags: int = 0):
    """One fused lora_apply call: y[:, slices] += delta of every projection."""
    abi.lora_apply(y, x, store.h_in, store.c_projs(), store.r_slot, store.n_slots, meta.c,
                   workspace, flags=flags, dev_status=dev_status, stream=stream)


def linear(y: torch.Tensor, x: torch.Tensor, W: torch.Tensor, store: GroupStore, meta: BatchMeta,
           workspace: torch.Tensor, dev_status=None, stream=None):
    """One lora_linear call: y[:, slices] = bf16(x W^T + delta) of every
    projection, W the group's stacked base weight [ld_y][h_in]."""
    abi.lora_linear(y, x, store.h_in, W, store.c_projs(), store.r_slot, store.n_slots, meta.c, workspace,
                    dev_status=dev_status, stream=stream)
