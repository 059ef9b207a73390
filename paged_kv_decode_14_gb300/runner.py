"""Device-side driver for one workload: upload, build the cache by append,
run decode steps.  Used by the tests, the smoke check and the benchmark."""

from __future__ import annotations

import numpy as np
import torch

from . import _native as nat
from .workloads import BF16_NAN, FP8_NAN, Workload


def _bf16_tensor(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


class DeviceWorkload:
    """Holds a workload's tensors on the GPU.  The cache starts filled with the
    NaN sentinel, so a read of an unwritten slot shows up as NaN."""

    # The per-step inputs, in the order they sit in one device buffer (`io`).
    IO_FIELDS = ("q", "k_new", "v_new", "slots", "block_tables", "context_lens", "q_lens")

    def __init__(self, w: Workload, device="cuda", num_ctas: int = 0):
        self.w = w
        self.device = torch.device(device)
        dev = self.device
        # One step's inputs live in one device buffer, each field at a 256-byte
        # aligned offset, so a serving loop (and the end-to-end benchmark)
        # uploads them with a single copy from a pinned host mirror.
        arrays = {"q": (w.q.view(np.int16), torch.bfloat16), "k_new": (w.k_new.view(np.int16), torch.bfloat16),
                  "v_new": (w.v_new.view(np.int16), torch.bfloat16), "slots": (w.slots, torch.int64),
                  "block_tables": (np.ascontiguousarray(w.block_tables), torch.int32),
                  "context_lens": (w.context_lens, torch.int32), "q_lens": (w.q_lens, torch.int32)}
        offs, total = {}, 0
        for n in self.IO_FIELDS:
            offs[n] = total
            total += -(-max(1, arrays[n][0].nbytes) // 256) * 256
        host = np.zeros(total, dtype=np.uint8)
        for n in self.IO_FIELDS:
            a = np.ascontiguousarray(arrays[n][0])
            host[offs[n]:offs[n] + a.nbytes] = a.reshape(-1).view(np.uint8)
        self.io_host = torch.from_numpy(host)
        self.io = self.io_host.to(dev)
        for n in self.IO_FIELDS:
            a, dt = arrays[n]
            view = self.io[offs[n]:offs[n] + a.nbytes].view(dt).view(a.shape)
            setattr(self, n, view)
        ks = vs = None
        if w.kv_dtype == "fp8":
            ks = torch.from_numpy(w.k_scales).to(dev)
            vs = torch.from_numpy(w.v_scales).to(dev)
        self.cache = nat.PagedKVCache(w.num_blocks, w.num_kv_heads, w.head_dim, w.kv_dtype, device=dev,
                                      k_scales=ks, v_scales=vs)
        self.reset_cache()
        self.num_ctas = num_ctas
        # the decode/verify kernels' workspace (their query windows are at most
        # 16 long; longer windows go to the prefill kernel, which needs none)
        self.workspace = None
        if max(1, w.max_q_len) <= 16:
            self.workspace = nat.make_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                                max(1, w.max_q_len), num_ctas, device=dev)
        self.append_err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.prefill_err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out = torch.empty_like(self.q)

    def pinned_io(self) -> torch.Tensor:
        """A pinned host copy of the step's input buffer (same layout as `io`)."""
        return self.io_host.pin_memory()

    def reset_cache(self):
        if self.w.kv_dtype == "fp8":
            self.cache.k.fill_(int(FP8_NAN))
            self.cache.v.fill_(int(FP8_NAN))
        else:
            self.cache.k.view(torch.int16).fill_(int(np.int16(BF16_NAN.view(np.int16))))
            self.cache.v.view(torch.int16).fill_(int(np.int16(BF16_NAN.view(np.int16))))

    def prefill(self, chunk_tokens: int = 1 << 16):
        """Append the workload's resident tokens (the state before the step)."""
        w = self.w
        n = int(w.prefill_slots.shape[0])
        for s in range(0, n, chunk_tokens):
            e = min(n, s + chunk_tokens)
            k = _bf16_tensor(w.prefill_k[s:e], self.device)
            v = _bf16_tensor(w.prefill_v[s:e], self.device)
            sl = torch.from_numpy(w.prefill_slots[s:e]).to(self.device)
            nat.append(self.cache, k, v, sl, device_error=self.append_err)

    def append_step(self, stream=None):
        nat.append(self.cache, self.k_new, self.v_new, self.slots, device_error=self.append_err, stream=stream)

    def attend(self, out=None, num_ctas=None, stream=None, workspace=None):
        w = self.w
        return nat.attention(self.cache, self.q, self.block_tables, self.context_lens, self.q_lens,
                             max(1, w.max_q_len), w.scale, workspace if workspace is not None else self.workspace,
                             out=self.out if out is None else out,
                             num_ctas=self.num_ctas if num_ctas is None else num_ctas, stream=stream)

    def attend_cascade(self, out=None, stream=None):
        """Attention with each shared-prefix group's prefix attended once
        (pkv_paged_attention_cascade); the groups come from the workload."""
        w = self.w
        if not hasattr(self, "cascade_ws"):
            gs, gp = w.prefix_groups()
            self.group_starts = torch.from_numpy(gs).to(self.device)
            self.group_prefix_lens = torch.from_numpy(gp).to(self.device)
            self.max_group_q = int(max(int(w.q_lens[gs[g]:gs[g + 1]].sum()) for g in range(len(gp))))
            self.cascade_ws = nat.make_cascade_workspace(w.num_seqs, len(gp), w.num_q_heads, w.num_kv_heads,
                                                         w.head_dim, max(1, w.max_q_len), self.max_group_q,
                                                         device=self.device)
        return nat.attention_cascade(self.cache, self.q, self.block_tables, self.context_lens, self.q_lens,
                                     max(1, w.max_q_len), self.group_starts, self.group_prefix_lens,
                                     self.max_group_q, w.scale, self.cascade_ws,
                                     out=self.out if out is None else out, stream=stream)

    def attend_prefill(self, out=None, stream=None):
        """Causal attention of the step's query windows on the chunked-prefill
        kernel (pkv_paged_prefill; bf16 caches, any window length)."""
        w = self.w
        return nat.prefill(self.cache, self.q, self.block_tables, self.context_lens, self.q_lens,
                           max(1, w.max_q_len), w.scale, out=self.out if out is None else out,
                           device_error=self.prefill_err, stream=stream)

    def step(self, stream=None):
        """One decode step: append the new tokens, then attend."""
        self.append_step(stream)
        return self.attend(stream=stream)

    def cache_bytes(self):
        """(K, V) cache contents as numpy arrays in the library layout."""
        k = self.cache.k.view(torch.uint8) if self.w.kv_dtype == "fp8" else self.cache.k.view(torch.int16)
        v = self.cache.v.view(torch.uint8) if self.w.kv_dtype == "fp8" else self.cache.v.view(torch.int16)
        k, v = k.cpu().numpy().reshape(-1), v.cpu().numpy().reshape(-1)
        if self.w.kv_dtype != "fp8":
            k, v = k.view(np.uint16), v.view(np.uint16)
        return k, v

    def errors(self):
        """(attention error bits: workspace and prefill words, append error
        bits); clears them.
        After a timeout the workspace may hold merge tickets of the aborted
        call: it is zeroed again, ready for the next call."""
        a = nat.read_device_error(self.prefill_err)
        if self.workspace is not None:
            ws = nat.read_device_error(self.workspace)
            if ws & nat.DEVERR_TIMEOUT:
                nat.workspace_init(self.workspace)
            a |= ws
        return a, nat.read_device_error(self.append_err)
