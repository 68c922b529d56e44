"""Token-sharded data parallelism of one linear layer's quantize-then-GEMM step.

Data parallelism gives each rank its own tokens: the rows of the activations X
[M, K] and of the gradients dY [M, N] are split across ranks, and every rank
holds the whole weight W [N, K].  Of the three GEMMs of a linear ("How to
optimize Transformer-based models for low-precision training", autocast vs
pre-quantize: Fprop, Dgrad, Wgrad), Fprop (Y = X W^T) and Dgrad (dX = dY W)
keep their rows on the rank; Wgrad (dW = dY^T X) reduces over the tokens, so
each rank computes a partial sum.  Lower precision also means fewer bytes to
exchange ("Faster training throughput in FP8 with NVIDIA NeMo", why speed-up
matters).  The step has two exchange steps, both through torch.distributed
(NCCL between GPUs, gloo on the CPU):

1. all-reduce MAX of the shard amaxes.  Per-tensor FP8 and NVFP4 scale every
   value of a tensor by one factor from the tensor's global amax ("Optimizing
   Transformer models for low-precision training", per-tensor scaling;
   "Accelerate LLM training with NVFP4 on Blackwell", FP32 tensor scale).  Each
   rank runs the amax pass (lpq_amax) on its shard, one all-reduce combines
   the few floats of all of the linear's tensors, and each rank quantizes with
   the global values (LPQ_GIVEN_AMAX): the codes and scales of a shard are then
   those of the same rows of the unsharded tensor.  The stochastic rounding of
   the row-wise dY copy keeps that property through its counter offset (first
   row x columns); the column-wise dY copy's counters follow the shard's own
   [N, M_shard] layout.  Delayed scaling reduces the amax its quantize pass
   measured before the history update, so every rank keeps the same state.
   The MX formats have block-local scales and need no amax exchange.
2. all-reduce SUM of the FP32 Wgrad partial dW_g = dY_g^T X_g.

Every computation runs in liblpq's CUDA kernels (through the C ABI binding);
this module only orders the calls and the two collectives.
"""
import torch

from . import lpq

# Recipes: quantizer (format, extra flags, scaling) per tensor role.
RECIPES = ("bf16", "fp8_current", "fp8_delayed", "mxfp8", "mxfp8_e5m2", "mxfp4", "nvfp4")


def shard_rows(total_rows, world, rank, granule=128):
    """Rows [r0, r1) of rank `rank` when `total_rows` tokens are split into
    `world` contiguous shards of whole `granule`-row groups (the last group
    may be short), as evenly as the groups allow."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank must be in [0, world)")
    groups = -(-total_rows // granule)
    base, extra = divmod(groups, world)
    g0 = rank * base + min(rank, extra)
    g1 = g0 + base + (1 if rank < extra else 0)
    return min(total_rows, g0 * granule), min(total_rows, g1 * granule)


def _dist():
    import torch.distributed as dist
    return dist if dist.is_available() and dist.is_initialized() else None


def exchange_amax(amax, group=None):
    """Exchange 1: in-place all-reduce MAX of a 1-D FP32 tensor of shard
    amaxes (several tensors' values in one call).  No-op without an
    initialized process group or with one rank."""
    dist = _dist()
    if dist is not None and dist.get_world_size(group) > 1:
        dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    return amax


def exchange_wgrad(dw, group=None):
    """Exchange 2: in-place all-reduce SUM of the FP32 Wgrad partials."""
    dist = _dist()
    if dist is not None and dist.get_world_size(group) > 1:
        dist.all_reduce(dw, op=dist.ReduceOp.SUM, group=group)
    return dw


def quant_config(recipe, role):
    """(format, extra flags, scaling) of tensor role X, W or dY under `recipe`:
    NVFP4 uses 16x16 tiles for W, stochastic rounding for dY and the Hadamard
    transform on the Wgrad operands (the column-wise copies of X and dY)."""
    L = lpq
    if recipe in ("fp8_current", "fp8_delayed"):
        fmt = L.FP8_E5M2 if role == "dY" else L.FP8_E4M3
        return fmt, 0, L.SCALING_DELAYED if recipe == "fp8_delayed" else L.SCALING_CURRENT
    if recipe == "mxfp8":
        return L.MXFP8, 0, L.SCALING_CURRENT
    if recipe == "mxfp8_e5m2":
        return (L.MXFP8_E5M2 if role == "dY" else L.MXFP8), 0, L.SCALING_CURRENT
    if recipe == "mxfp4":
        return L.MXFP4, 0, L.SCALING_CURRENT
    if recipe == "nvfp4":
        if role == "W":
            return L.NVFP4_2D, 0, L.SCALING_CURRENT
        extra = L.STOCHASTIC if role == "dY" else 0
        return L.NVFP4, extra | L.RHT_COLWISE, L.SCALING_CURRENT
    raise ValueError(recipe)


class TokenShardedLinear:
    """One linear's Fprop, Dgrad and Wgrad on this rank's token shard.

    X [m, K] and dY [m, N] are this rank's rows (its first row has global index
    `first_row`), W [N, K] the replicated weight.  step() quantizes every
    tensor once into both copies (amax exchange first where the recipe needs
    it), runs the three GEMMs into Y [m, N], dX [m, K] (bf16) and the FP32
    Wgrad partial, and all-reduces dW over the group."""

    def __init__(self, recipe, X, W, dY, first_row=0, group=None, rht_seed=1234):
        if recipe not in RECIPES:
            raise ValueError(recipe)
        self.recipe, self.X, self.W, self.dY = recipe, X, W, dY
        self.first_row, self.group, self.rht_seed = int(first_row), group, rht_seed
        dev = X.device
        m, K = X.shape
        N = W.shape[0]
        self.m, self.K, self.N = m, K, N
        self.Y = torch.empty((m, N), dtype=torch.bfloat16, device=dev)
        self.dX = torch.empty((m, K), dtype=torch.bfloat16, device=dev)
        self.dW = torch.empty((N, K), dtype=torch.float32, device=dev)
        L = lpq
        both = L.ROWWISE | L.COLWISE
        self.q = {}
        self.states = {}
        if recipe == "bf16":
            return
        for role, t in (("X", X), ("W", W), ("dY", dY)):
            fmt, _, scaling = quant_config(recipe, role)
            self.q[role] = L.alloc(fmt, t.shape[0], t.shape[1], both, L.SF_GEMM, dev)
            if scaling == L.SCALING_DELAYED:
                self.states[role] = L.DelayedState(16, dev)
        # The amaxes the exchange combines, one FP32 slot each: the views'
        # amax fields point into this buffer, so the amax passes write it and
        # the quantizers read it in place.
        self.global_amax = recipe in ("fp8_current", "fp8_delayed", "nvfp4")
        if self.global_amax:
            self.amax = torch.zeros(4, dtype=torch.float32, device=dev)
            for i, (role, copy) in enumerate((("X", "row"), ("X", "col"), ("dY", "row"), ("dY", "col"))):
                getattr(self.q[role], copy).amax = self.amax[i:i + 1]

    def _quantize(self, role, t, flags, seed, counter_offset=0):
        L = lpq
        fmt, extra, scaling = quant_config(self.recipe, role)
        st = self.states.get(role)
        L.quantize(t, fmt, flags | extra, scaling=scaling, seed=seed, counter_offset=counter_offset,
                   rht_seed=self.rht_seed, state=st, out=self.q[role])

    def quantize_all(self, seed=0):
        """Both copies of X, W and dY, with the amax exchange where needed."""
        L = lpq
        both = L.ROWWISE | L.COLWISE
        r = self.recipe
        ctr = self.first_row * self.N  # dY row-wise SR counters continue the global row-major order
        if r == "fp8_delayed":
            # the quantize pass measures the shard amax (fused) with the scale of
            # the earlier steps; the global amax then feeds the history update
            self._quantize("W", self.W, both, seed)
            self._quantize("X", self.X, both, seed)
            self._quantize("dY", self.dY, both, seed, ctr)
            a = torch.stack([self.q["X"].row.amax[0], self.q["dY"].row.amax[0]])
            exchange_amax(a, self.group)
            for i, role in enumerate(("X", "dY")):
                fmt = quant_config(r, role)[0]
                L.scale_update(self.states[role], a[i:i + 1], L.FMAX[fmt])
            L.scale_update(self.states["W"], self.q["W"].row.amax, L.FMAX[L.FP8_E4M3])
            return
        self._quantize("W", self.W, both, seed)  # replicated: its own amax, no exchange
        if self.global_amax:
            rht = r == "nvfp4"
            L.amax(self.X, rht=rht, rht_seed=self.rht_seed, out=self.amax[0:1], rht_out=self.amax[1:2] if rht else None)
            L.amax(self.dY, rht=rht, rht_seed=self.rht_seed, out=self.amax[2:3],
                   rht_out=self.amax[3:4] if rht else None)
            if not rht:  # per-tensor FP8: one amax for both copies
                self.amax[1:2].copy_(self.amax[0:1])
                self.amax[3:4].copy_(self.amax[2:3])
            exchange_amax(self.amax, self.group)
            self._quantize("X", self.X, both | L.GIVEN_AMAX, seed)
            self._quantize("dY", self.dY, both | L.GIVEN_AMAX, seed, ctr)
        else:
            self._quantize("X", self.X, both, seed)
            self._quantize("dY", self.dY, both, seed, ctr)

    def step(self, seed=0):
        """Quantize, Fprop, Dgrad, Wgrad partial, all-reduce SUM of dW."""
        L = lpq
        if self.recipe == "bf16":
            L.gemm(L.FPROP, L.Copy.of_bf16(self.X), L.Copy.of_bf16(self.W), c=self.Y)
            L.gemm(L.DGRAD, L.Copy.of_bf16(self.dY), L.Copy.of_bf16(self.W.t().contiguous(), True), c=self.dX)
            L.gemm(L.WGRAD, L.Copy.of_bf16(self.dY.t().contiguous(), True),
                   L.Copy.of_bf16(self.X.t().contiguous(), True), c=self.dW, out_fp32=True)
        else:
            self.quantize_all(seed)
            q = self.q
            L.gemm(L.FPROP, q["X"].row, q["W"].row, c=self.Y)
            L.gemm(L.DGRAD, q["dY"].row, q["W"].col, c=self.dX)
            L.gemm(L.WGRAD, q["dY"].col, q["X"].col, c=self.dW, out_fp32=True)
        exchange_wgrad(self.dW, self.group)
        return self.Y, self.dX, self.dW
