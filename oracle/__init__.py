"""CPU oracle for partition-guided online structured FFN pruning (POP).

TEST INFRASTRUCTURE ONLY. This package is the slow, plain statement of what
the GPU library computes. Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it; the
library itself never calls it and has no CPU fallback.

It shares no code with the CUDA path (no kernels, headers, helpers, tables or
constant generators). Inputs come from the ``synth`` package, which only draws
random numbers.

Arithmetic is float64 with library primitives (matmul, sqrt, sort) as steps.
Where floating point decides a set (the R/C/P partition, the per-step top-k),
the decision is taken on float32 keys, the precision the GPU kernels use, so
that both sides decide in the same precision.

Sources (cited by page title and section):

* [POP] "POP: Online Structural Pruning Enables Efficient Inference of Large
  Foundation Models", papernotes.org NeurIPS 2026 notes: "Overall framework",
  "Key design 1" (importance and the three regions), "Key design 2" (decode
  partial forward, candidate scoring, top-k fill), "Key design 3" (FFN-only
  pruning, 29.9% FFN rate), "Loss / training strategy" (gamma = 0.1, about 20%
  candidates, Wanda metric, partition at the first forward).
* [BWAP] "Batch-wise adaptive pruning: periodic neuron-activation-aware weight
  pruning for language reasoning models", bittide page: Section 3.1 eq. (1)
  (gated MLP), abstract and Fig. 2(a) (element-wise max batch aggregation,
  periodic top-k with activation memory).

Readings where the pages are silent or garbled (each repeated at its function):

1. Importance (Key design 1 prints ||W_{:,i} (.) s||_2 with s_k = ||X_{:,:,k}||_2,
   dimension-inconsistent): W is the down projection W2, i an intermediate
   channel, s_i = ||Z_{:,:,i}||_2 over all B*L prompt tokens, so
   I_i = ||W2[:, i]||_2 * s_i (the Wanda form named under "Loss / training").
2. delta = gamma; quantile cut-offs are counts, rounded half-to-even:
   n_P = round(max(0, r - gamma) * N), n_R = N - round(min(1, r + gamma) * N),
   keep = N - round(r * N), k = keep - n_R.
3. Ties at every cut-off go to the lower channel index (ranked as more
   important).
4. Decode score of candidate i: max over the batch of |z_{b,i}| * ||W2[:, i]||
   (element-wise max aggregation, [BWAP] Fig. 2(a)); for B = 1 this is the
   single-token Wanda score.
5. Prefill itself runs dense; masking starts at the first decode step.
6. Periodic variant (the [BWAP] text stops before its score definition): the
   memory M sums the aggregated candidate scores every step; at steps with
   t mod P == 0 the selection is redone from M and M is cleared; in between
   the last selection is held. P = 1 is per-step POP.
7. MoE experts ([POP] "Loss / training strategy" applies the method to MoE
   models with dynamic routing, taking the partition at the first forward,
   but gives no routing rule): each token goes to its two largest router
   logits (ties to the lower expert), weighted by the softmax over those two
   logits. Each expert's partition comes from the prompt tokens routed to it;
   an expert that gets none has s = 0, so I = 0 and the index tie rule alone
   decides its split. Every decode step advances every expert's step counter
   and memory; an expert that receives no token in a step scores each
   candidate 0 (the maximum of non-negative values over no tokens) and
   contributes no output.
8. Periodic "skip" variant (the [BWAP] abstract's periodic top-k read so that
   the mask's saving reaches the gate/up too): at update steps (t mod P == 0)
   the step is the full one above; in between, gate/up runs only over R and
   the held selection S, the memory gains the scores of S only (the other
   candidates are not computed) and y is the same sum over R u S. P = 1 is
   per-step POP.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "silu", "ffn_activations", "dense_ffn", "column_norms", "channel_importance", "RegionCounts",
    "region_counts", "partition", "candidate_scores", "select_topk", "down_projection", "prefill",
    "PopSession", "moe_route", "moe_prefill", "MoeSession", "moe_decode",
]


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def silu(v: np.ndarray) -> np.ndarray:
    """SiLU(v) = v * sigmoid(v) = v / (1 + exp(-v))  ([BWAP] Section 3.1, the sigma of eq. (1))."""
    v = _f64(v)
    return v / (1.0 + np.exp(-v))


def ffn_activations(Wg, W1, X) -> np.ndarray:
    """FF activations z = SiLU(Wg x) (.) (W1 x) for every token (row) of X.

    [BWAP] Section 3.1, eq. (1): Wg, W1 in R^{D_FF x D}; X is [T, D]; returns
    Z [T, D_FF] in float64.
    """
    X = _f64(X)
    G = X @ _f64(Wg).T
    U = X @ _f64(W1).T
    return silu(G) * U


def down_projection(W2, Z, channels=None) -> np.ndarray:
    """FF2(z) = W2 z restricted to the given channels ([BWAP] Section 3.1; [POP] flowchart, last box).

    y_b = sum over i in `channels` (ascending) of z_{b,i} * W2[:, i]. With
    channels = all of [0, D_FF) this is the dense output.
    """
    W2 = _f64(W2)
    Z = _f64(Z)
    if channels is None:
        channels = np.arange(W2.shape[1])
    channels = np.sort(np.asarray(channels, dtype=np.int64))
    return Z[:, channels] @ W2[:, channels].T


def dense_ffn(Wg, W1, W2, X) -> np.ndarray:
    """Dense gated MLP: Y = W2 (SiLU(Wg x) (.) W1 x) per token ([BWAP] Section 3.1)."""
    Z = ffn_activations(Wg, W1, X)
    return down_projection(W2, Z)


def column_norms(W2) -> np.ndarray:
    """||W2[:, i]||_2 for every intermediate channel i (the weight factor of the Wanda score)."""
    W2 = _f64(W2)
    return np.sqrt(np.sum(W2 * W2, axis=0))


def channel_importance(W2, Z):
    """Prefill importance of each intermediate channel ([POP] Key design 1; "Loss / training strategy").

    ss_i = sum over all prompt tokens of z_i^2, s_i = sqrt(ss_i),
    I_i = ||W2[:, i]||_2 * s_i   (reading 1 in the module docstring).
    Returns (ss, I) in float64.
    """
    Z = _f64(Z)
    ss = np.sum(Z * Z, axis=0)
    I = column_norms(W2) * np.sqrt(ss)
    return ss, I


@dataclass(frozen=True)
class RegionCounts:
    N: int
    n_P: int
    n_R: int
    n_C: int
    keep: int
    k: int


def _round_half_even(v: float) -> int:
    return int(round(v))  # Python's round() on a float is round-half-to-even


def region_counts(N: int, r: float, gamma: float) -> RegionCounts:
    """Sizes of the three regions and of the per-step fill ([POP] Key design 1 and 2).

    tau_low = q_{r - delta}, tau_high = q_{r + delta} with delta = gamma
    (reading 2). The survivors per step number (1 - r) * N ("|R| plus the
    selected candidates match the survivor count the global rate asks for").
    """
    if not (0.0 <= r <= 1.0) or gamma < 0.0 or N < 0:
        raise ValueError("need 0 <= r <= 1, gamma >= 0, N >= 0")
    n_P = _round_half_even(max(0.0, r - gamma) * N)
    n_R = N - _round_half_even(min(1.0, r + gamma) * N)
    keep = N - _round_half_even(r * N)
    k = keep - n_R
    n_C = N - n_P - n_R
    if not (0 <= k <= n_C):
        raise ValueError(f"fill count k={k} outside [0, |C|={n_C}]")
    return RegionCounts(N=N, n_P=n_P, n_R=n_R, n_C=n_C, keep=keep, k=k)


def partition(I, counts: RegionCounts):
    """Three-way split of the channels by prefill importance ([POP] Key design 1).

    Channels are ordered from least to most important by (I ascending, index
    descending), so that among equal scores the lower index counts as more
    important (reading 3). P = the first n_P (at or below tau_low), R = the
    last n_R (at or above tau_high), C = the rest (strictly between).
    The decision is taken on float32 keys. Returns (R, C, P), each ascending.
    """
    key = np.asarray(I, dtype=np.float32)
    N = key.shape[0]
    assert N == counts.N
    idx = np.arange(N)
    order = np.lexsort((-idx, key))  # primary: key ascending; secondary: index descending
    P = np.sort(order[:counts.n_P])
    C = np.sort(order[counts.n_P:N - counts.n_R])
    R = np.sort(order[N - counts.n_R:])
    return R, C, P


def candidate_scores(Z_C, n2_C) -> np.ndarray:
    """Per-step score of each candidate ([POP] Key design 2; [BWAP] Fig. 2(a)).

    a_i = max over the batch of |z_{b,i}| * ||W2[:, i]||  (reading 4).
    Z_C is [B, |C|], n2_C is [|C|]. Returns float64.
    """
    Z_C = _f64(Z_C)
    if Z_C.shape[1] == 0:
        return np.zeros(0)
    if Z_C.shape[0] == 0:  # no token this step (an idle MoE expert, reading 7)
        return np.zeros(Z_C.shape[1])
    return np.max(np.abs(Z_C), axis=0) * _f64(n2_C)


def select_topk(scores, k: int) -> np.ndarray:
    """Positions of the k largest scores ([POP] Key design 2: sort descending, take the top).

    Decided on float32 keys; ties go to the lower position (reading 3).
    Returns the selected positions in ascending order.
    """
    key = np.asarray(scores, dtype=np.float32)
    n = key.shape[0]
    if not (0 <= k <= n):
        raise ValueError("k outside [0, n]")
    pos = np.arange(n)
    order = np.lexsort((pos, -key))  # primary: key descending; secondary: position ascending
    return np.sort(order[:k])


def prefill(Wg, W1, W2, X, r: float, gamma: float):
    """Prefill: dense forward over the prompt, importance, and the R/C/P split.

    [POP] Overall framework and Key design 1; prefill runs dense (reading 5).
    Returns a dict with Y (dense output), ss, I, counts and R, C, P.
    """
    Z = ffn_activations(Wg, W1, X)
    Y = down_projection(W2, Z)
    ss, I = channel_importance(W2, Z)
    counts = region_counts(_f64(W2).shape[1], r, gamma)
    R, C, P = partition(I, counts)
    return dict(Y=Y, Z=Z, ss=ss, I=I, counts=counts, R=R, C=C, P=P)


@dataclass
class PopSession:
    """Decode-time state of one layer ([POP] Key design 2; [BWAP] abstract, periodic top-k and memory).

    Holds the partition (R, C ascending), the fill count k, the update period P
    and the activation memory M over C (reading 6). `step()` runs one decode
    step on x_t [B, D] and returns y_t [B, D].
    """
    Wg: np.ndarray
    W1: np.ndarray
    W2: np.ndarray
    R: np.ndarray
    C: np.ndarray
    k: int
    period: int = 1
    skip: bool = False   # reading 8: between updates, gate/up only over R u S
    t: int = 0
    memory: np.ndarray = field(default=None)
    S: np.ndarray = field(default=None)          # selected candidate positions (into C), ascending
    last_scores: np.ndarray = field(default=None)
    last_z: np.ndarray = field(default=None)

    def __post_init__(self):
        self.Wg = _f64(self.Wg)
        self.W1 = _f64(self.W1)
        self.W2 = _f64(self.W2)
        self.R = np.asarray(self.R, dtype=np.int64)
        self.C = np.asarray(self.C, dtype=np.int64)
        if self.period < 1:
            raise ValueError("period must be >= 1")
        if not (0 <= self.k <= self.C.shape[0]):
            raise ValueError("k outside [0, |C|]")
        self.n2_C = column_norms(self.W2[:, self.C]) if self.C.size else np.zeros(0)
        self.memory = np.zeros(self.C.shape[0])

    def step(self, x) -> np.ndarray:
        x = _f64(x)
        if self.skip and self.t % self.period != 0:
            return self._skip_step(x)
        RC = np.concatenate([self.C, self.R])
        # H_t = f(X_t; R u C): gate/up only over the retained and candidate rows
        Z_RC = ffn_activations(self.Wg[RC], self.W1[RC], x)
        Z_C = Z_RC[:, :self.C.shape[0]]
        a = candidate_scores(Z_C, self.n2_C)
        self.memory = self.memory + a
        if self.t % self.period == 0:
            self.S = select_topk(self.memory, self.k)
            self.memory = np.zeros_like(self.memory)
        self.last_scores = a
        self.last_z = Z_RC
        self.t += 1
        # final FFN over R and the selected candidates, ascending channel order
        keep = np.sort(np.concatenate([self.R, self.C[self.S]]))
        Z_full = np.zeros((x.shape[0], self.W2.shape[1]))
        Z_full[:, RC] = Z_RC
        return down_projection(self.W2, Z_full, keep)

    def _skip_step(self, x) -> np.ndarray:
        """A step between updates of the skip variant (reading 8): z over R and the held S only."""
        CS = self.C[self.S]
        RS = np.concatenate([CS, self.R])
        Z_RS = ffn_activations(self.Wg[RS], self.W1[RS], x)
        a_S = candidate_scores(Z_RS[:, :CS.shape[0]], self.n2_C[self.S])
        self.memory[self.S] = self.memory[self.S] + a_S
        self.last_scores = np.zeros(self.C.shape[0])
        self.last_scores[self.S] = a_S
        self.last_z = Z_RS
        self.t += 1
        keep = np.sort(np.concatenate([self.R, CS]))
        Z_full = np.zeros((x.shape[0], self.W2.shape[1]))
        Z_full[:, RS] = Z_RS
        return down_projection(self.W2, Z_full, keep)

    def kept_channels(self) -> np.ndarray:
        """Channel indices used by the last step's down projection (R plus the selected candidates)."""
        return np.sort(np.concatenate([self.R, self.C[self.S]]))


def moe_route(logits, top: int = 2):
    """Top-`top` routing of MoE tokens with softmax weights over the selected logits.

    [POP] "Loss / training strategy" names MoE dynamic routing without a rule;
    this takes the common top-2 gate. Ties go to the lower expert. Returns
    (experts [T, top] int64, weights [T, top] float64).
    """
    L = _f64(logits)
    T, E = L.shape
    e_idx = np.arange(E)
    experts = np.empty((T, top), dtype=np.int64)
    for t in range(T):
        order = np.lexsort((e_idx, -L[t]))
        experts[t] = order[:top]
    sel = np.take_along_axis(L, experts, axis=1)
    w = np.exp(sel - sel.max(axis=1, keepdims=True))
    w /= w.sum(axis=1, keepdims=True)
    return experts, w


def _routed_tokens(experts, e: int) -> np.ndarray:
    """Ascending indices of the tokens whose routing includes expert e."""
    return np.nonzero(np.any(experts == e, axis=1))[0]


def _combine(experts, weights, outputs, D: int) -> np.ndarray:
    """y_t = sum over the token's routing choices j (in rank order) of w_{t,j} * (expert e_{t,j}'s output for t).

    `outputs[e]` maps token index -> that expert's output row.
    """
    T = experts.shape[0]
    Y = np.zeros((T, D))
    for t in range(T):
        for j in range(experts.shape[1]):
            Y[t] += weights[t, j] * outputs[int(experts[t, j])][t]
    return Y


def moe_prefill(expert_weights, X, logits, r: float, gamma: float, top: int = 2):
    """Prefill of an MoE layer of gated-MLP experts (reading 7).

    expert_weights: list of (Wg, W1, W2) per expert; X [T, D]; logits [T, E].
    Each expert runs `prefill` on its routed tokens (ascending token order) and
    takes its partition from them; the layer output is the routing-weighted sum
    of the experts' dense outputs. Returns dict(Y, experts, weights, parts) with
    parts[e] = dict(R, C, P, I, counts, tokens).
    """
    X = _f64(X)
    experts, weights = moe_route(logits, top)
    D = X.shape[1]
    outputs, parts = [], []
    for e, (Wg, W1, W2) in enumerate(expert_weights):
        tok = _routed_tokens(experts, e)
        N = _f64(Wg).shape[0]
        if tok.size:
            pre = prefill(Wg, W1, W2, X[tok], r, gamma)
            parts.append(dict(R=pre["R"], C=pre["C"], P=pre["P"], I=pre["I"], counts=pre["counts"], tokens=tok))
            outputs.append({int(t): pre["Y"][row] for row, t in enumerate(tok)})
        else:
            counts = region_counts(N, r, gamma)
            I = np.zeros(N)
            R, C, P = partition(I, counts)
            parts.append(dict(R=R, C=C, P=P, I=I, counts=counts, tokens=tok))
            outputs.append({})
    return dict(Y=_combine(experts, weights, outputs, D), experts=experts, weights=weights, parts=parts)


@dataclass
class MoeSession:
    """Decode-time state of an MoE layer: one PopSession per expert (reading 7).

    `step(x, logits)` routes the B tokens, runs every expert's decode step on the
    tokens routed to it (possibly none) and combines the outputs.
    """
    sessions: list
    top: int = 2
    last_experts: np.ndarray = field(default=None)
    last_weights: np.ndarray = field(default=None)

    def step(self, x, logits) -> np.ndarray:
        x = _f64(x)
        experts, weights = moe_route(logits, self.top)
        outputs = []
        for e, sess in enumerate(self.sessions):
            tok = _routed_tokens(experts, e)
            ye = sess.step(x[tok])
            outputs.append({int(t): ye[row] for row, t in enumerate(tok)})
        self.last_experts, self.last_weights = experts, weights
        return _combine(experts, weights, outputs, x.shape[1])


def moe_decode(expert_weights, parts, xs, logits, k: int, period: int = 1, top: int = 2):
    """The decode steps of an MoE layer, expert by expert (the same results as MoeSession.step).

    expert_weights(e) -> (Wg, W1, W2) loads one expert's weights, so that only one expert's float64
    copy is alive at a time; parts[e] = dict(R, C) is its partition; xs[t] [B, D] and logits[t]
    [B, E] are the steps' inputs. The experts' steps are independent of one another, so running
    each expert through all steps before the next gives the same outputs as stepping the layer.
    Returns (ys [T, B, D], per_expert) with per_expert[e] = list over steps of dict(S, scores, C).
    """
    T = len(xs)
    routes = [moe_route(l, top) for l in logits]
    outputs = [[] for _ in range(T)]
    per_expert = []
    for e, part in enumerate(parts):
        sess = PopSession(*expert_weights(e), part["R"], part["C"], k, period=period)
        steps = []
        for t in range(T):
            tok = _routed_tokens(routes[t][0], e)
            ye = sess.step(_f64(xs[t])[tok])
            outputs[t].append({int(tt): ye[row] for row, tt in enumerate(tok)})
            steps.append(dict(S=sess.C[sess.S], scores=sess.last_scores, C=sess.C))
        per_expert.append(steps)
        del sess
    D = _f64(xs[0]).shape[1]
    ys = np.stack([_combine(routes[t][0], routes[t][1], outputs[t], D) for t in range(T)])
    return ys, per_expert
