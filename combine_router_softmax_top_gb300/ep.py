"""Expert-parallel (EP) exchange of the MoE layer between ranks: the count
exchange and the all-to-allv of the send buffer that the standard all-to-all
dispatcher performs (the MoE expert-parallel overlap skill card, section "what
it is", dispatcher table; EP16 in its benchmark sections), and the mirrored
return of the expert outputs.

Each rank owns E/R experts (rank d owns experts d*E/R .. (d+1)*E/R - 1). A
rank's dispatch layout (moe_dispatch_layout / moe_dispatch_fused with R ranks)
already writes its send buffer rank-major and expert-contiguous, with the
per-(rank, local expert) counts cnt_re [R, E/R] and the chunk starts
rank_off [R+1]. The exchange is then:
  1. counts:  every rank sends cnt_re[d] to rank d and receives recv_cnt [R, E/R],
     recv_cnt[s] = source s's cnt_re[this rank] (an all-to-all of R*E/R ints);
  2. rows:    an all-to-allv of the send buffer with send splits
     rank_off[d+1] - rank_off[d] and receive splits recv_cnt.sum(1); rows
     arrive in source order ("receive order");
  3. the receiver re-sorts them expert-major on the GPU (moe_ep_resort) before
     its expert GEMMs, and back to receive order before the return exchange,
     which is step 2 with the splits swapped.
This module is communication plumbing over torch.distributed (NCCL on GPUs,
gloo on CPU): it moves buffers and reads the split sizes to the host (the
all-to-allv needs them there); all arithmetic stays in the CUDA kernels.
"""
from __future__ import annotations

from typing import List, Optional, Tuple

import torch
import torch.distributed as dist


def send_splits(rank_off: torch.Tensor) -> List[int]:
    """Rows this rank sends to each rank: rank_off[d+1] - rank_off[d]."""
    ro = rank_off.detach().to("cpu", torch.int64)
    return (ro[1:] - ro[:-1]).tolist()


def recv_splits(recv_cnt: torch.Tensor) -> List[int]:
    """Rows this rank receives from each source: recv_cnt.sum(1)."""
    return recv_cnt.detach().to("cpu", torch.int64).sum(1).tolist()


def exchange_counts(cnt_re: torch.Tensor, group: Optional[dist.ProcessGroup] = None
                    ) -> torch.Tensor:
    """Count exchange: cnt_re [R, E/R] int32 (rows to rank d's local expert l)
    -> recv_cnt [R, E/R] int32 (rows from source s for this rank's local expert l)."""
    R = dist.get_world_size(group)
    if cnt_re.dim() != 2 or cnt_re.shape[0] != R:
        raise ValueError(f"cnt_re must be [R={R}, E/R], got {tuple(cnt_re.shape)}")
    send = cnt_re.contiguous()
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv.view(-1), send.view(-1), group=group)
    return recv


def exchange_rows(send: torch.Tensor, splits_out: List[int], splits_in: List[int],
                  group: Optional[dist.ProcessGroup] = None) -> torch.Tensor:
    """All-to-allv of rows: send [sum(splits_out), H] (chunk d goes to rank d)
    -> [sum(splits_in), H] (chunk s came from rank s)."""
    if send.shape[0] < sum(splits_out):
        raise ValueError(f"send has {send.shape[0]} rows, the splits need {sum(splits_out)}")
    src = send[:sum(splits_out)].contiguous()
    recv = send.new_empty((sum(splits_in),) + tuple(send.shape[1:]))
    dist.all_to_all_single(recv, src, output_split_sizes=splits_in,
                           input_split_sizes=splits_out, group=group)
    return recv


def dispatch(send: torch.Tensor, cnt_re: torch.Tensor, rank_off: torch.Tensor,
             group: Optional[dist.ProcessGroup] = None
             ) -> Tuple[torch.Tensor, torch.Tensor, List[int], List[int]]:
    """Count exchange then row exchange of one layer's send buffer.
    Returns (recv rows in receive order, recv_cnt, splits sent, splits received)."""
    recv_cnt = exchange_counts(cnt_re, group)
    out_s, in_s = send_splits(rank_off), recv_splits(recv_cnt)
    return exchange_rows(send, out_s, in_s, group), recv_cnt, out_s, in_s


def combine_return(back: torch.Tensor, splits_sent: List[int], splits_received: List[int],
                   group: Optional[dist.ProcessGroup] = None) -> torch.Tensor:
    """The mirrored exchange: rows in receive order go back to their sources,
    which get them in their own send-buffer order (the layout slot[] indexes)."""
    return exchange_rows(back, splits_received, splits_sent, group)
