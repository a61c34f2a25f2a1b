"""CPU oracle for the data-parallel optimizer step of DDP, ZeRO-1/2/3 and the FSDP unit.

TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the cpu_baseline /
reference leg of bench.py may import or run this module. The CUDA library neither imports
it nor shares any code, header, table or constant generator with it; the only shared
module is `synth` (seeded inputs, no arithmetic of the method).

Plain, slow and written to be checked by eye against the pages:
  [Wiring]     "Behind the scenes of distributed training, and why your GPU wiring matters as
               much as your strategy" (automationscribe.com), Part 1.
  [Interview]  "DP、ZeRO-1/2/3、FSDP:每卡显存多少、通信多多少?" (charliedreemur.github.io,
               ml-interview / dp-zero-fsdp).
  [Concepts]   "Data Parallel, ZeRO and FSDP" (k8ai.app, concepts / parallelism / data-parallel).

Precision. The pages fix the step's precision: bf16 param and grad, fp32 master / m / v
([Interview] "先弄清楚" DDP item: 16 bytes per parameter; [Concepts] "Limits of plain DP").
So the reduction and Adam run in float32 here, one IEEE-rounded numpy operation per
arithmetic step, in the order written below (numpy never fuses a multiply into an add).
The FSDP linear reference is computed in float64 and rounded once.

Readings where the pages are silent (the same readings the CUDA library's header states):
  * reduced gradient = (((g_0 + g_1) + g_2) + ... + g_{N-1}) in fp32, rank order, then
    multiplied by f32(1/N); it stays fp32 (never rounded to bf16).
  * Adam = Kingma & Ba with bias correction, eps outside the square root, decoupled weight
    decay; the exact op sequence is in `adam_update`.
  * bias corrections 1 - beta^t are evaluated in binary64 (C pow) and rounded to fp32.
  * bf16 rounding is round-to-nearest-even; NaN stays NaN.
  * layout: psi padded to a multiple of N, contiguous rank-major shards, buckets of
    C = floor(bucket_bytes / (2N)) elements in every rank's shard.

Parity status: every function here is pinned by tests/test_oracle_pins.py (closed forms
and worked numbers printed on the pages, invariants the pages state, library routines for
special cases, brute force on tiny inputs). No function is "parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F32 = np.float32


# ========================================================================================
# bf16 <-> fp32
# ========================================================================================

def bf16_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns -> float32. A bf16 value is the upper 16 bits of a binary32,
    so widening is exact: put the 16 bits on top and zero the rest."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16(x) -> np.ndarray:
    """float32 -> bf16 bit patterns, IEEE round-to-nearest, ties to even, on the 16 dropped
    bits. A carry out of the kept mantissa moves to the next binade (and past the largest
    finite value to infinity), exactly as IEEE rounding requires. NaN -> quiet NaN."""
    xf = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = xf.view(np.uint32)
    hi = u >> np.uint32(16)
    lo = u & np.uint32(0xFFFF)
    half = np.uint32(0x8000)
    round_up = (lo > half) | ((lo == half) & ((hi & np.uint32(1)) == 1))
    nan = np.isnan(xf)
    out = np.where(nan, hi | np.uint32(0x0040), hi + round_up.astype(np.uint32))
    return out.astype(np.uint16)


# ========================================================================================
# flat-buffer layout: padding, shards, buckets
# ========================================================================================

@dataclass(frozen=True)
class Layout:
    """Flat parameter / gradient / state buffer of psi elements shared out to N ranks.

    [Interview] "ZeRO-1 / 2 / 3": model states are cut into N parts by data-parallel rank,
    each card keeps and updates only its 1/N. [Interview] follow-up "FSDP2 和 FSDP1": FSDP1
    flattens and concatenates parameters into one flat parameter before cutting it.
    Padding to a multiple of N makes the N parts equal; padding entries stay zero.
    """
    psi: int
    n_ranks: int
    bucket_bytes: int
    psi_padded: int
    shard: int
    bucket_elems: int
    n_buckets: int


def make_layout(psi: int, n_ranks: int, bucket_bytes: int) -> Layout:
    if psi < 1 or n_ranks < 1:
        raise ValueError("psi and n_ranks must be >= 1")
    if bucket_bytes < 2 * n_ranks:
        raise ValueError("a bucket must hold at least one bf16 element per rank")
    psi_padded = ((psi + n_ranks - 1) // n_ranks) * n_ranks
    shard = psi_padded // n_ranks
    # a bucket of bucket_bytes bf16 gradient bytes spans all N rank segments, so each
    # rank's shard contributes bucket_bytes / (2N) elements to it
    bucket_elems = bucket_bytes // (2 * n_ranks)
    n_buckets = (shard + bucket_elems - 1) // bucket_elems
    return Layout(psi, n_ranks, bucket_bytes, psi_padded, shard, bucket_elems, n_buckets)


def shard_range(lay: Layout, rank: int):
    """Flat index range [lo, hi) owned by `rank`."""
    return rank * lay.shard, (rank + 1) * lay.shard


def bucket_range(lay: Layout, rank: int, k: int):
    """Flat index range of bucket k inside rank's shard."""
    base = rank * lay.shard
    return base + k * lay.bucket_elems, base + min((k + 1) * lay.bucket_elems, lay.shard)


def owner(lay: Layout, j: int) -> int:
    return j // lay.shard


# ========================================================================================
# simulated collectives (N ranks = N arrays held by this process)
# ========================================================================================

def inv_n(n_ranks: int):
    """f32(1/N): the fp32 number nearest 1/N (one correctly rounded fp32 division)."""
    return F32(1.0) / F32(n_ranks)


def as_f32(x) -> np.ndarray:
    """A gradient contribution as fp32: bf16 bit patterns (uint16) are widened exactly,
    fp32 arrays (the Megatron distributed optimizer's fp32 gradients) are taken as they are."""
    a = np.asarray(x)
    if a.dtype == np.uint16:
        return bf16_to_f32(a)
    if a.dtype != np.float32:
        raise TypeError(f"gradient contributions are bf16 bits or fp32, not {a.dtype}")
    return a


def reduce_sum_scale(grads, lo: int, hi: int) -> np.ndarray:
    """The reduced gradient for flat indices [lo, hi): the N ranks' contributions (bf16,
    or fp32 for the Megatron distributed optimizer) in fp32, added one rank at a time in
    rank order 0..N-1, then scaled by 1/N to the average ([Wiring] DDP section: the GPUs
    average their gradients; [Concepts] "Plain data parallel (DDP)" step 2)."""
    n = len(grads)
    acc = as_f32(grads[0][lo:hi]).copy()
    for q in range(1, n):
        acc = acc + as_f32(grads[q][lo:hi])
    return acc * inv_n(n)


def reduce_scatter(lay: Layout, grads, rank: int) -> np.ndarray:
    """Reduce-scatter: sums everyone's gradients but hands each rank only its own slice of
    the sum ([Wiring] "ZeRO: The Dial Between DDP and FSDP"; [Interview] "reduce-scatter 与
    all-gather"). Done bucket by bucket; the bucket split never changes a value."""
    out = np.empty(lay.shard, dtype=np.float32)
    base = rank * lay.shard
    for k in range(lay.n_buckets):
        lo, hi = bucket_range(lay, rank, k)
        out[lo - base:hi - base] = reduce_sum_scale(grads, lo, hi)
    return out


def all_gather(shards) -> np.ndarray:
    """All-gather: the N slices concatenated in rank order into one full copy."""
    return np.concatenate(list(shards))


def all_reduce(lay: Layout, grads) -> np.ndarray:
    """All-reduce, by definition: every flat element j gets the rank-order fp32 sum of the
    N contributions times 1/N. The pages state that this equals a reduce-scatter followed
    by an all-gather; the pin tests check that against `reduce_scatter` + `all_gather`."""
    return reduce_sum_scale(grads, 0, lay.psi_padded)


# ========================================================================================
# mixed-precision Adam
# ========================================================================================

@dataclass(frozen=True)
class AdamHyper:
    """Adam hyper-parameters; each is used as the nearest float32."""
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0


def bias_corrections(hp: AdamHyper, t: int):
    """(1 - beta1^t, 1 - beta2^t): powers of the fp32 betas taken in binary64 with C pow,
    subtracted from one in binary64, each rounded once to fp32. t counts from 1."""
    if t < 1:
        raise ValueError("Adam step counts from 1")
    b1 = float(F32(hp.beta1))
    b2 = float(F32(hp.beta2))
    return F32(1.0 - math.pow(b1, t)), F32(1.0 - math.pow(b2, t))


def adam_update(master, m, v, g, hp: AdamHyper, t: int, return_update: bool = False):
    """One Adam step on fp32 master / m / v with fp32 gradient g; returns new arrays
    (master, m, v[, u]) where u is the update term subtracted from master.

    The pages fix the state (fp32 master, momentum and variance; [Wiring] "Take Mistral-7B
    and fine-tune it with Adam"; [Interview] DDP item) but not the equations, so this is
    Kingma & Ba's Adam with bias correction, eps outside the square root and decoupled
    weight decay, each line one fp32 operation:
        m  = beta1*m + (1-beta1)*g
        v  = beta2*v + (1-beta2)*(g*g)
        mh = m / (1-beta1^t);   vh = v / (1-beta2^t)
        den = sqrt(vh) + eps
        master = master - (lr*wd)*master          (only when wd != 0)
        u = lr * (mh / den);    master = master - u
    """
    b1, b2 = F32(hp.beta1), F32(hp.beta2)
    omb1, omb2 = F32(1.0) - b1, F32(1.0) - b2
    lr, eps, wd = F32(hp.lr), F32(hp.eps), F32(hp.weight_decay)
    bc1, bc2 = bias_corrections(hp, t)
    g = np.asarray(g, dtype=np.float32)
    m_new = b1 * np.asarray(m, dtype=np.float32) + omb1 * g
    v_new = b2 * np.asarray(v, dtype=np.float32) + omb2 * (g * g)
    mh = m_new / bc1
    vh = v_new / bc2
    den = np.sqrt(vh) + eps
    w = np.asarray(master, dtype=np.float32)
    if wd != F32(0.0):
        lr_wd = lr * wd
        w = w - lr_wd * w
    u = lr * (mh / den)
    w = w - u
    if return_update:
        return w, m_new, v_new, u
    return w, m_new, v_new


def fused_step_elements(grads_at, master, m, v, hp: AdamHyper, t: int):
    """The whole per-element step for a set of flat indices, as plain composition:
    reduced gradient -> Adam -> bf16 cast. `grads_at` is a list of N bf16 arrays holding
    each rank's contribution at those indices. Returns (master, m, v, param_bf16)."""
    g = reduce_sum_scale(grads_at, 0, len(grads_at[0]))
    w, m1, v1 = adam_update(master, m, v, g, hp, t)
    return w, m1, v1, f32_to_bf16(w)


# ========================================================================================
# what each rank holds, per strategy
# ========================================================================================

STAGES = ("ddp", "zero1", "zero2", "zero3", "megatron")
STAGE_IDS = {"ddp": 0, "zero1": 1, "zero2": 2, "zero3": 3}


def rank_buffer_shapes(stage: str, lay: Layout):
    """Elements and dtype of every model-state buffer one rank keeps between steps.

    [Interview] Fig. 1 and "手算例子:7B、N = 8"; [Concepts] "ZeRO and FSDP" stage table:
      DDP     param 2P   grad 2P   master/m/v 12P          (full everything)
      ZeRO-1  param 2P   grad 2P   master/m/v 12P/N        (optimizer state sharded)
      ZeRO-2  param 2P   grad 2P/N master/m/v 12P/N        (+ gradients)
      ZeRO-3  param 2P/N grad 2P/N master/m/v 12P/N        (+ parameters)
      Megatron distributed optimizer: bf16 param 2P, fp32 grad 4P, master/m/v 12P/N.
    P is the padded length; the N incoming gradient chunks and the fp32 reduced gradient
    are transient simulation buffers and are not model state.
    """
    P, S = lay.psi_padded, lay.shard
    bf16, f32 = np.uint16, np.float32
    if stage == "ddp":
        return {"param": (P, bf16), "grad": (P, bf16), "master": (P, f32), "m": (P, f32), "v": (P, f32)}
    if stage == "zero1":
        return {"param": (P, bf16), "grad": (P, bf16), "master": (S, f32), "m": (S, f32), "v": (S, f32)}
    if stage == "zero2":
        return {"param": (P, bf16), "grad": (S, bf16), "master": (S, f32), "m": (S, f32), "v": (S, f32)}
    if stage == "zero3":
        return {"param": (S, bf16), "grad": (S, bf16), "master": (S, f32), "m": (S, f32), "v": (S, f32)}
    if stage == "megatron":
        return {"param": (P, bf16), "grad": (P, f32), "master": (S, f32), "m": (S, f32), "v": (S, f32)}
    raise ValueError(stage)


def model_state_bytes(stage: str, lay: Layout):
    """Bytes per rank of each held buffer, from `rank_buffer_shapes`, plus the total."""
    out = {}
    for name, (n, dt) in rank_buffer_shapes(stage, lay).items():
        out[name] = n * np.dtype(dt).itemsize
    out["total"] = sum(out.values())
    return out


def comm_elements(stage: str, lay: Layout, zero1_via_allreduce: bool = False):
    """Elements each rank moves per step, per collective ([Interview] "每卡通信量";
    [Concepts] stage table):
      DDP: all-reduce = reduce-scatter P + all-gather P            -> 2P
      ZeRO-1 / ZeRO-2: reduce-scatter P + all-gather of params P    -> 2P
      ZeRO-1 implemented with a gradient all-reduce then a param all-gather -> 3P
        ([Interview] follow-up on ZeRO-1 vs ZeRO-2 communication)
      ZeRO-3 / FSDP: all-gather fwd P + all-gather bwd P + reduce-scatter P -> 3P
    Ring algorithms multiply each by (N-1)/N (`ring_sent_elements`)."""
    P = lay.psi_padded
    if stage in ("ddp", "megatron"):
        c = {"reduce_scatter": P, "all_gather_fwd": P, "all_gather_bwd": 0}
    elif stage == "zero1" and zero1_via_allreduce:
        c = {"reduce_scatter": P, "all_gather_fwd": 2 * P, "all_gather_bwd": 0}
    elif stage in ("zero1", "zero2"):
        c = {"reduce_scatter": P, "all_gather_fwd": P, "all_gather_bwd": 0}
    elif stage == "zero3":
        c = {"reduce_scatter": P, "all_gather_fwd": P, "all_gather_bwd": P}
    else:
        raise ValueError(stage)
    c["total"] = c["reduce_scatter"] + c["all_gather_fwd"] + c["all_gather_bwd"]
    return c


def ring_sent_elements(elements: int, n_ranks: int) -> int:
    """A ring collective over P elements sends N-1 chunks of P/N per rank."""
    assert elements % n_ranks == 0
    return (n_ranks - 1) * (elements // n_ranks)


def ring_allreduce_bytes(grad_bytes: float, n_ranks: int) -> float:
    """Per-GPU bytes sent (and received) by a ring all-reduce of grad_bytes:
    2 (N-1)/N * S ([Concepts] "Communication cost")."""
    return 2.0 * (n_ranks - 1) / n_ranks * grad_bytes


# ========================================================================================
# the step, rank by rank, for every strategy
# ========================================================================================

@dataclass
class RankState:
    stage: str
    rank: int
    buffers: dict = field(default_factory=dict)

    def nbytes(self):
        return sum(a.nbytes for a in self.buffers.values())


def init_ranks(stage: str, lay: Layout, master0: np.ndarray):
    """Every rank's buffers before step 1: master from the fp32 init (full or own shard),
    m = v = 0, bf16 param = RNE(master) (full, or own shard under ZeRO-3), grads zero."""
    ranks = []
    param_full = f32_to_bf16(master0)
    for r in range(lay.n_ranks):
        shapes = rank_buffer_shapes(stage, lay)
        b = {name: np.zeros(n, dtype=dt) for name, (n, dt) in shapes.items()}
        lo, hi = shard_range(lay, r)
        b["master"][:] = master0 if stage == "ddp" else master0[lo:hi]
        b["param"][:] = param_full[lo:hi] if stage == "zero3" else param_full
        ranks.append(RankState(stage, r, b))
    return ranks


def step_ranks(ranks, lay: Layout, local_grads, hp: AdamHyper, t: int):
    """One optimizer step of every rank. local_grads[q] is rank q's full bf16 gradient
    from its own backward pass (length P).

    DDP ([Concepts] "Plain data parallel (DDP)"): all-reduce, then the identical Adam on
    every full replica.
    ZeRO-1/2 ([Interview] "ZeRO-1 / 2 / 3"; "每卡通信量"): reduce-scatter bucket by bucket,
    Adam on the own 1/N of master/m/v, all-gather of the updated bf16 params into every
    rank's full param buffer. ZeRO-2 keeps only its own slice of the gradient.
    ZeRO-3: as ZeRO-2, but each rank keeps only its own bf16 param slice; the full
    parameters exist only when `gather_params` assembles them for a unit.
    Megatron distributed optimizer ([Interview] worked table, Megatron row and the note
    beneath it): full bf16 params and full fp32 gradients (local_grads are fp32), fp32
    master / m / v sharded; reduce-scatter, shard Adam and param all-gather as ZeRO-1.
    """
    stage = ranks[0].stage
    n = lay.n_ranks
    for r, st in enumerate(ranks):
        lo, hi = shard_range(lay, r)
        st.buffers["grad"][:] = local_grads[r] if st.buffers["grad"].size == lay.psi_padded else local_grads[r][lo:hi]
    if stage == "ddp":
        g_full = all_reduce(lay, local_grads)
        for st in ranks:
            b = st.buffers
            b["master"], b["m"], b["v"] = adam_update(b["master"], b["m"], b["v"], g_full, hp, t)
            b["param"] = f32_to_bf16(b["master"])
        return ranks
    new_shards = []
    for r, st in enumerate(ranks):
        b = st.buffers
        g_shard = reduce_scatter(lay, local_grads, r)
        b["master"], b["m"], b["v"] = adam_update(b["master"], b["m"], b["v"], g_shard, hp, t)
        new_shards.append(f32_to_bf16(b["master"]))
    if stage in ("zero1", "zero2", "megatron"):
        full = all_gather(new_shards)
        for st in ranks:
            st.buffers["param"] = full.copy()
    elif stage == "zero3":
        for r, st in enumerate(ranks):
            st.buffers["param"] = new_shards[r]
    else:
        raise ValueError(stage)
    return ranks


def gather_params(ranks) -> np.ndarray:
    """The full bf16 parameter buffer as rank 0 sees it after the step (ZeRO-3: the
    all-gather of every rank's slice, which FSDP performs per unit before use)."""
    if ranks[0].stage == "zero3":
        return all_gather([st.buffers["param"] for st in ranks])
    return ranks[0].buffers["param"]


def gather_master(ranks, lay: Layout) -> np.ndarray:
    if ranks[0].stage == "ddp":
        return ranks[0].buffers["master"]
    return all_gather([st.buffers["master"] for st in ranks])


# ========================================================================================
# FSDP unit: gather row shards, then the linear that consumes them
# ========================================================================================

def gather_rows(shards) -> np.ndarray:
    """[Interview] follow-up "手写 FSDP 的一层 linear": each card stores 1/N of W's rows;
    before use the full W is all-gathered: row-concatenation in rank order (a bit copy)."""
    return np.concatenate([np.asarray(s) for s in shards], axis=0)


def fsdp_linear_forward(a_bf16, w_shards_bf16):
    """Forward of the FSDP linear on the local batch: Y = A W^T with W in the [out, in]
    layout of a linear layer, W gathered from its row shards.
    Returns (Y in float64, Y rounded to fp32, Y in bf16 = RNE of the fp32 Y).
    float64 holds every bf16 x bf16 product exactly; only the sum is rounded."""
    a = bf16_to_f32(a_bf16).astype(np.float64)
    w = bf16_to_f32(gather_rows(w_shards_bf16)).astype(np.float64)
    y64 = a @ w.T
    y32 = y64.astype(np.float32)
    return y64, y32, f32_to_bf16(y32)


def fsdp_linear_backward(a_bf16, w_shards_bf16, dy_bf16, n_ranks: int):
    """Backward of the FSDP linear ([Interview] follow-up on a hand-written FSDP linear):
    all-gather W again, dX = dY W, the full-shape dW = dY^T A, then dW is reduce-scattered
    so each rank keeps its 1/N of the rows. Here one rank's batch is given; the reduced
    dW over N ranks whose contributions are dW_q is `reduce_rows` below.
    Returns (dX float64, dW float64)."""
    a = bf16_to_f32(a_bf16).astype(np.float64)
    w = bf16_to_f32(gather_rows(w_shards_bf16)).astype(np.float64)
    dy = bf16_to_f32(dy_bf16).astype(np.float64)
    return dy @ w, dy.T @ a


def reduce_rows(dw_list, n_ranks: int, rank: int) -> np.ndarray:
    """Reduce-scatter of full-shape weight gradients over dim 0: rank keeps rows
    [rank*R/N, (rank+1)*R/N) of the rank-order sum times 1/N (fp32, like `reduce_sum_scale`)."""
    rows = dw_list[0].shape[0]
    assert rows % n_ranks == 0
    rs = rows // n_ranks
    acc = np.asarray(dw_list[0][rank * rs:(rank + 1) * rs], dtype=np.float32).copy()
    for q in range(1, len(dw_list)):
        acc = acc + np.asarray(dw_list[q][rank * rs:(rank + 1) * rs], dtype=np.float32)
    return acc * inv_n(len(dw_list))


# ========================================================================================
# full MLP unit (Mistral-style): gate / up projections, SiLU-gate product, down projection
# ========================================================================================

def silu(x):
    """SiLU (swish): x * sigmoid(x) = x / (1 + exp(-x)), in float64."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def mlp_unit_forward(x_bf16, gate_shards, up_shards, down_shards=None, h_bf16=None):
    """The MLP unit an FSDP wrap of a Mistral-style block computes on its local batch, each
    weight gathered from its row shards first ([Interview] Fig. 2: gather, compute, free):
        G = X W_gate^T,  U = X W_up^T,  H = silu(G) * U,  Y = H W_down^T.
    Everything in float64. Returns (G, U, H, Y); Y is computed from `h_bf16` (the bf16 H a
    kernel produced, an exact input to the next product) when given, else from H, and is
    None without down_shards."""
    x = bf16_to_f32(x_bf16).astype(np.float64)
    g = x @ bf16_to_f32(gather_rows(gate_shards)).astype(np.float64).T
    u = x @ bf16_to_f32(gather_rows(up_shards)).astype(np.float64).T
    h = silu(g) * u
    y = None
    if down_shards is not None:
        hin = h if h_bf16 is None else bf16_to_f32(h_bf16).astype(np.float64)
        y = hin @ bf16_to_f32(gather_rows(down_shards)).astype(np.float64).T
    return g, u, h, y


def silu_gate_backward(dh_bf16, g_bf16, u_bf16):
    """Backward of H = silu(G) * U (the MLP unit's SiLU-gate product; [Interview] Fig. 2:
    the unit's backward after its forward) from the activations the forward saved and the
    upstream dH, all bf16, in float64:
        s = 1 / (1 + exp(-g)),  silu(g) = g s,  silu'(g) = s (1 + g (1 - s)),
        dU = dH silu(G),  dG = dH U silu'(G).
    Returns (dG, dU) in float64."""
    dh = bf16_to_f32(dh_bf16).astype(np.float64)
    g = bf16_to_f32(g_bf16).astype(np.float64)
    u = bf16_to_f32(u_bf16).astype(np.float64)
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-g))
    return dh * u * (s * (1.0 + g * (1.0 - s))), dh * (g * s)


def transpose_cat(srcs) -> np.ndarray:
    """The FSDP backward's operand layout: dst[c][q*rows + r] = srcs[q][r][c] — the sources
    transposed and placed side by side (W^T from W's row shards is the backward all-gather,
    [Interview] follow-up on a hand-written FSDP linear). A bit copy."""
    return np.concatenate([np.asarray(s).T for s in srcs], axis=1)
