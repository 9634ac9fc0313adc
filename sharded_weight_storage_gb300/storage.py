"""Device-memory plumbing over PyTorch for the C library: allocates the N
chunk buffers of every layer, the two slots, the scale tensors and the
workspace, runs the one-time relayout from row shards, and creates the
context. Every step of the path itself runs in libsws.so kernels."""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import torch

from . import _lib as L


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    return (stream or torch.cuda.current_stream()).cuda_stream


class ShardedStack:
    """Resident storage for a plan: chunk (l, i) is its own device buffer,
    standing in for rank i's shard of layer l."""

    def __init__(self, entries: Sequence[tuple], n_shards: int, max_m: int = 64, device: str = "cuda",
                 flags: int = 0):
        """flags: plan flags (L.SCALES_IN_T puts each sharded E4M3 entry's
        block scales into T right after the weight)."""
        self.plan = L.Plan(entries, n_shards, flags)
        self.flags = flags
        self.entries = list(entries)
        self.n_layers, self.n_shards, self.n_entries = self.plan.info()
        self.device = torch.device(device)
        self.layout = [self.plan.layer(l) for l in range(self.n_layers)]
        self.entry_info = [self.plan.entry(j) for j in range(self.n_entries)]
        self.scale_info = [self.plan.scales(j) for j in range(self.n_entries)]  # (offset in T or -1, bytes)
        self.chunks: List[List[Optional[torch.Tensor]]] = []
        for total, chunk, _ in self.layout:
            self.chunks.append([torch.empty(chunk, dtype=torch.uint8, device=self.device) if total else None
                                for _ in range(n_shards)])
        sb = self.plan.slot_bytes
        self.slots = [torch.empty(max(sb, 16), dtype=torch.uint8, device=self.device) for _ in range(2)]
        self.scales: List[Optional[torch.Tensor]] = [None] * self.n_entries
        self.replicated: List[Optional[torch.Tensor]] = [None] * self.n_entries
        self.max_m = max_m
        self.workspace = torch.empty(L.workspace_bytes(self.plan, max_m), dtype=torch.uint8, device=self.device)
        self.ctx: Optional[L.Ctx] = None

    # -- loading ---------------------------------------------------------------
    def layer_entries(self, layer: int) -> List[int]:
        return [j for j, e in enumerate(self.entries) if e[0] == layer]

    def load_layer(self, layer: int, codes: Dict[int, torch.Tensor], scales: Dict[int, torch.Tensor],
                   stream: Optional[torch.cuda.Stream] = None):
        """codes[j]: full weight bytes of entry j (host or device, uint8 [rows,
        cols*elem]); they are cut into the loader's 1/N row shards on the device
        and relaid into this layer's chunks by the relayout kernel.
        scales[j]: float32 block scales [ceil(rows/128), ceil(cols/128)] of an
        E4M3 entry, or one number - a per-tensor scale (ModelOpt FP8), kept
        replicated outside T and stored as that grid filled with it; absent for
        BF16 and F16 entries."""
        n = self.n_shards
        shard_ptrs, keep = [], []
        for j in self.layer_entries(layer):
            off, nbytes, sharded = self.entry_info[j]
            w = codes[j].to(self.device, non_blocking=False).contiguous()
            sc = scales.get(j)
            if sc is not None:
                _, _, rows, cols = self.entries[j]
                grid = (-(-rows // 128), -(-cols // 128))
                if not torch.is_tensor(sc):
                    sc = torch.tensor(sc, dtype=torch.float32)
                if sc.numel() == 1 and tuple(sc.shape) != grid:
                    sc = torch.full(grid, float(sc.reshape(-1)[0]), dtype=torch.float32)
                self.scales[j] = sc.to(self.device, dtype=torch.float32).contiguous()
            if not sharded:
                self.replicated[j] = w
                continue
            rows = w.shape[0]
            parts = [w[r * (rows // n):(r + 1) * (rows // n)].contiguous() for r in range(n)]
            keep += parts
            shard_ptrs += [p.data_ptr() for p in parts]
        if self.layout[layer][0] == 0:
            return
        chunk_ptrs = [c.data_ptr() for c in self.chunks[layer]]
        L.relayout(self.plan, layer, shard_ptrs, chunk_ptrs, _stream_ptr(stream))
        if any(self.scale_info[j][0] >= 0 for j in self.layer_entries(layer)):
            # scales in T: each chunk takes its window of the full scale tensors
            L.relayout_scales(self.plan, layer, [self.scales[j].data_ptr() if self.scale_info[j][0] >= 0 else 0
                                                 for j in self.layer_entries(layer)], chunk_ptrs, _stream_ptr(stream))
        (stream or torch.cuda.current_stream()).synchronize()
        del keep

    def make_ctx(self) -> L.Ctx:
        chunk_ptrs = [c.data_ptr() if c is not None else 0 for row in self.chunks for c in row]
        self.ctx = L.Ctx(self.plan, chunk_ptrs, self.slots[0].data_ptr(), self.slots[1].data_ptr(),
                         [s.data_ptr() if s is not None else 0 for s in self.scales],
                         [r.data_ptr() if r is not None else 0 for r in self.replicated],
                         self.workspace.data_ptr(), self.workspace.numel())
        return self.ctx

    # -- accounting -------------------------------------------------------------
    def resident_chunk_bytes(self) -> int:
        return sum(c.numel() for row in self.chunks for c in row if c is not None)

    def slot_scales(self, slot: int, j: int) -> torch.Tensor:
        """Entry j's block scales inside a slot (scales-in-T layout)."""
        off, nbytes = self.scale_info[j]
        _, _, rows, cols = self.entries[j]
        return self.slots[slot][off:off + nbytes].view(torch.float32).view(-(-rows // 128), -(-cols // 128))

    def slot_view(self, slot: int, j: int) -> torch.Tensor:
        off, nbytes, sharded = self.entry_info[j]
        layer, _, rows, cols = self.entries[j]
        return self.slots[slot][off:off + nbytes].view(rows, -1)
