"""Expert parallelism for the MoE layer: the experts split across ranks, the routed rows
exchanged with all-to-all.

AngelSlim mcore_qad walkthrough (nxmr.cn/news/131691), section 二.4: the routed experts are
split across ranks only by expert parallelism (ETP = 1), so every expert's weight matrices stay
whole on one rank and the E experts are partitioned E / EP per rank (the ModelOpt QAD skill
page, "Choose topology explicitly": num_experts % EP == 0).  Section 二.5: scale gradients of
replicated parameters are averaged over their data-parallel group; for the experts that is the
expert-data-parallel group (the ranks that hold the same experts).

One step, each rank holding its own tokens:

  forward   1. plan: every valid (token, slot) pair (expert in [0, E), not a repeat of an
               earlier slot's expert -- the layer's own routing rule) goes to the rank that
               owns its expert, e // (E / EP); pairs leave in (destination, token, slot) order;
            2. all-to-all of the pairs' x rows and local expert ids;
            3. the owner runs the layer on the received rows with top-1 routing and weight 1,
               so its output rows are the expert outputs Y (received rows of one expert keep
               (source rank, token, slot) order: the order a single process would give the
               ranks' tokens concatenated);
            4. all-to-all back; out[t] = bf16(sum_j p[t, j] Y[t, j]) on the sending rank.
  backward  5. all-to-all of the pairs' dout rows and routing weights to the owners;
            6. the owners' input-gradient call with those weights (the layer's own dY =
               bf16(p dout), dprobs = <dout, Y> and dA1 rows), all-to-all of dA1 and dprobs
               back, and dx[t] = bf16(sum_j dA1[t, j]) on the sending rank;
            7. the owners' scale-gradient call (their experts only), averaged over the
               expert-data-parallel group.

The arithmetic runs in a backend: CudaExperts (the library's C ABI on this rank's GPU) in the
product.  The exchange itself is host logic over torch.distributed (NCCL on GPUs).
"""
import torch
import torch.distributed as dist


def _world(group):
    return dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1


def _rank(group):
    return dist.get_rank(group) if dist.is_available() and dist.is_initialized() else 0


def valid_pairs(topk_idx, E):
    """[T, k] bool: the pairs the layer keeps -- expert in [0, E) and not a repeat of an earlier
    slot's expert in the same token (the later slot is dropped)."""
    idx = topk_idx.long()
    T, k = idx.shape
    ok = (idx >= 0) & (idx < E)
    for j in range(1, k):
        dup = (idx[:, :j] == idx[:, j:j + 1]).any(dim=1)
        ok[:, j] &= ~dup
    return ok


def make_plan(topk_idx, E, ep_size):
    """Where each pair goes.  Returns a dict:
      order        int64 [n_sent]: the flat pair ids t * k + j in sending order (destination
                   rank, then pair id);
      send_counts  list of ep_size ints: pairs sent to each rank;
      local_expert int32 [n_sent]: the expert of each sent pair, numbered on its owner;
      row_of       int32 [T, k]: the position t * k + j of each kept pair in the pair-ordered
                   buffers, -1 for a dropped pair."""
    if E % ep_size:
        raise ValueError("the expert count %d is not a multiple of the expert-parallel size %d" % (E, ep_size))
    e_loc = E // ep_size
    T, k = topk_idx.shape
    ok = valid_pairs(topk_idx, E).reshape(-1)
    idx = topk_idx.reshape(-1).long()
    dest = torch.where(ok, idx // e_loc, torch.full_like(idx, ep_size))  # dropped pairs sort last, unsent
    order = torch.argsort(dest, stable=True)
    n_sent = int(ok.sum())
    order = order[:n_sent]
    send_counts = torch.bincount(dest[ok], minlength=ep_size).tolist()
    local_expert = (idx[order] - dest[order] * e_loc).to(torch.int32)
    flat = torch.arange(T * k, device=topk_idx.device, dtype=torch.int32)
    row_of = torch.where(ok, flat, torch.full_like(flat, -1)).reshape(T, k).contiguous()
    return {"order": order, "send_counts": send_counts, "local_expert": local_expert, "row_of": row_of}


def exchange(t, send_counts, recv_counts, group):
    """all-to-all of the rows of t ([n, ...], grouped by destination rank in rank order)."""
    if _world(group) == 1:
        return t
    out = t.new_empty((sum(recv_counts),) + tuple(t.shape[1:]))
    # an empty tensor may carry any strides (a zero-row view, or one made from an empty array):
    # give it a fresh buffer so that the byte view below is valid
    send, recv = (t.contiguous() if t.shape[0] else t.new_empty(t.shape)), out
    if t.dtype == torch.bfloat16:  # moved as raw bytes (not every backend has bf16 or int16)
        send, recv = send.view(torch.uint8), out.view(torch.uint8)
    dist.all_to_all_single(recv, send, output_split_sizes=list(recv_counts), input_split_sizes=list(send_counts),
                           group=group)
    return out


def exchange_counts(send_counts, group, device):
    if _world(group) == 1:
        return list(send_counts)
    s = torch.tensor(send_counts, dtype=torch.int64, device=device)
    r = torch.empty_like(s)
    dist.all_to_all_single(r, s, group=group)
    return r.tolist()


class ExpertParallelMoE:
    """The MoE layer with its E experts split over the ranks of `group` (E / size each; this
    rank owns experts [rank * E / size, (rank + 1) * E / size)).  `backend` holds this rank's
    experts and does the arithmetic (CudaExperts).  `expert_dp_group`: the ranks holding the same
    experts, over which the scale gradients are averaged (None: no replication)."""

    def __init__(self, backend, E, group=None, expert_dp_group=None):
        self.backend = backend
        self.E = E
        self.group = group
        self.expert_dp_group = expert_dp_group
        self.ep = _world(group)
        if E % self.ep:
            raise ValueError("num_experts %% EP must be 0 (E = %d, EP = %d)" % (E, self.ep))
        self.first_expert = _rank(group) * (E // self.ep)
        self.plan = None

    def forward(self, x, topk_idx, topk_w):
        T, k = topk_idx.shape
        plan = make_plan(topk_idx, self.E, self.ep)
        recv_counts = exchange_counts(plan["send_counts"], self.group, x.device)
        pair_token = plan["order"] // k
        x_rows = exchange(x[pair_token], plan["send_counts"], recv_counts, self.group)
        e_rows = exchange(plan["local_expert"], plan["send_counts"], recv_counts, self.group)
        y_rows = self.backend.forward(x_rows, e_rows)
        y_back = exchange(y_rows, recv_counts, plan["send_counts"], self.group)
        y_pairs = y_back.new_zeros((T * k,) + tuple(y_back.shape[1:]))
        y_pairs[plan["order"]] = y_back
        out = self.backend.combine(y_pairs, plan["row_of"], topk_w)
        plan["recv_counts"] = recv_counts
        self.plan, self.topk_w = plan, topk_w
        return out

    def backward(self, dout):
        """dx [T, d] and dprobs [T, k] for the tokens of the last forward."""
        plan = self.plan
        T, k = plan["row_of"].shape
        send, recv = plan["send_counts"], plan["recv_counts"]
        g_rows = exchange(dout[plan["order"] // k], send, recv, self.group)
        p_rows = exchange(self.topk_w.reshape(-1)[plan["order"]].contiguous(), send, recv, self.group)
        da_rows, dp_rows = self.backend.dgrad(g_rows, p_rows)
        da_back = exchange(da_rows, recv, send, self.group)
        dp_back = exchange(dp_rows, recv, send, self.group)
        da_pairs = da_back.new_zeros((T * k,) + tuple(da_back.shape[1:]))
        da_pairs[plan["order"]] = da_back
        dprobs = dp_back.new_zeros(T * k)
        dprobs[plan["order"]] = dp_back
        dx = self.backend.combine(da_pairs, plan["row_of"], None)
        return dx, dprobs.reshape(T, k)

    def scale_grads(self):
        """ds13 [E / EP, 2F, d / B], ds2 [E / EP, d, F / B] of this rank's experts, averaged over
        the expert-data-parallel group."""
        ds13, ds2 = self.backend.scalegrad()
        n = _world(self.expert_dp_group) if self.expert_dp_group is not None else 1
        if n > 1:
            for g in (ds13, ds2):
                dist.all_reduce(g, op=dist.ReduceOp.SUM, group=self.expert_dp_group)
                g.div_(n)
        return ds13, ds2


class CudaExperts:
    """This rank's experts on its GPU, through the library's C ABI: w13 [E_loc, 2F, d], w2
    [E_loc, d, F] (bf16) and their scales; `flags` as for the layer calls."""

    def __init__(self, w13, s13, w2, s2, fmt, flags=0):
        import scale_only_quantization_gb300 as Q
        self.Q = Q
        self.w13, self.s13, self.w2, self.s2 = w13, s13, w2, s2
        self.fmt, self.flags = fmt, flags
        self.E_loc, twoF, self.d = w13.shape
        self.F = twoF // 2

    def forward(self, x_rows, local_expert):
        Q = self.Q
        n = x_rows.shape[0]
        self.s = Q.shape(n, self.d, self.F, self.E_loc, 1, self.fmt, self.flags)
        self.ws = torch.empty(Q.qad_moe_workspace_bytes(self.s), dtype=torch.uint8, device=x_rows.device)
        self.idx = local_expert.reshape(n, 1).contiguous()
        self.p = torch.ones((n, 1), dtype=torch.float32, device=x_rows.device)
        y = torch.empty((n, self.d), dtype=torch.bfloat16, device=x_rows.device)
        Q.qad_moe_fwd(self.s, x_rows.contiguous(), self.idx, self.p, self.w13, self.s13, self.w2, self.s2, y, self.ws)
        return y

    def dgrad(self, dout_rows, p_rows):
        """dA1 rows and dprobs of the received pairs: the layer's input-gradient call on the rows'
        output gradients with the pairs' routing weights."""
        n = dout_rows.shape[0]
        da = torch.empty_like(dout_rows)
        dp = torch.empty((n, 1), dtype=torch.float32, device=dout_rows.device)
        self.Q.qad_moe_bwd_dgrad(self.s, dout_rows.contiguous(), p_rows.reshape(n, 1).contiguous(), self.w13,
                                 self.s13, self.w2, self.s2, da, dp, self.ws)
        return da, dp.reshape(n)

    def scalegrad(self):
        ds13, ds2 = torch.empty_like(self.s13), torch.empty_like(self.s2)
        self.Q.qad_moe_bwd_scalegrad(self.s, self.w13, self.s13, self.w2, self.s2, ds13, ds2, 0, self.ws)
        return ds13, ds2

    def combine(self, rows, row_of, p):
        T, k = row_of.shape
        out = torch.empty((T, rows.shape[1]), dtype=torch.bfloat16, device=rows.device)
        self.Q.qad_moe_combine(rows.contiguous(), row_of, p, out, T, k, rows.shape[1])
        return out
