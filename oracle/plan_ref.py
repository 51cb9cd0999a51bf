"""Restatement of the plan rules of the library, for a bit-exact metadata check.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages fix what plan() is for, not how it partitions work: it builds helper
structures once for many later runs ("flashinfer.sparse", BlockSparseAttentionWrapper.plan
notes) and the MLA scheduler metadata is reusable
while seq_lens, the query shape and top-k stay unchanged ("Sparse MLA",
get_batch_decode_metadata_mla). The partition rule below is the library's own design,
stated here from its specification so that the C++ plan can be compared word for word:

Metadata = 16 header words
    magic 0x766b7362, kind (1 decode, 2 bsr, 3 mla), units, workers, chunks, slots,
    merges, tile, off_workers, off_chunks, off_merges, off_aux0, off_aux1, grid,
    total_words, variant
followed by sections, each starting at a multiple of 4 words (zero padding):
    worker_ptr[workers + 1], chunks[chunks][4], merges[merges][3], aux0, aux1.

Linear partition (decode, MLA). Units have lengths len_u (tokens); tiles_u =
ceil(len_u / tile); NT = sum of tiles; P = min(max_workers, NT); worker w owns the
global tiles [floor(w NT / P), floor((w+1) NT / P)), cut at unit boundaries into
chunks (unit, tok_begin, tok_end, slot) with tok_end clipped to len_u. A unit cut into
>= 2 chunks gives each chunk a partial-state slot, numbered in chunk order; otherwise
slot = -1. Merge items (unit, first_slot, count) list, in unit order, the units with
0 chunks (first_slot = -1) or >= 2 chunks.
  * decode: G = decode_group_heads(num_kv_heads, page_size). G > 0 (page_size <= 16
    and num_kv_heads <= 8 or a multiple of 8): variant 1, units (b, group of G kv
    heads) b-major, max_workers = num_sms unless given, grid = P, and instead of equal
    ranges the cost partition (linear_partition_cost with the costs of _fill, 2 tiles for a
    piece published mid-stream and 2 for a merge at the worker's end: the smallest bound T
    whose greedy left-to-right fill needs at most max_workers workers; P = the workers that
    fill uses). Otherwise variant 0,
    units (b, kv head) b-major, max_workers = 8 * num_sms unless given,
    grid = ceil(P / 8). Both: len = request length, tile 16, aux0 = kv_indptr,
    aux1 = kv_indices. Variant 1 appends, after the sections (total_words updated), one
    16-word start record per worker for the first chunk of its walk (its last chunk when it
    has several, else its only one): unit, first token, end token, slot, kv_indptr[b],
    pages of b, n = min(8, pages of b - first token // page_size), 0, and the first n page
    ids of that chunk (zeros after).
  * MLA: units = query tokens n = b*q_len + t, len = seq_lens[b], tile 128,
    max_workers = max(1, num_sms // 2) (a worker is a pair of CTAs, one per latent half),
    grid = 2 P, no aux, variant 0. Whole units instead of the linear partition when, with
    the units of at least one tile placed by longest processing time (tiles descending,
    stable; least-loaded worker, lowest index on ties) on G = min(max_workers, such units)
    workers, the busiest worker holds at most 7 tiles more than ceil(NT / P): chunks (u, 0,
    len_u, -1) per worker in assignment order, no slots, merge items (u, -1, 0) for the units
    without rows; P = G then.
  * variable-block BSR (variant 2): per kv head h and row block a, in that order, a
    descriptor (first query token, row count, first tile, end tile); the tiles split each
    maximal run of consecutive visible column blocks [s, e) into (t, e) for t = s, s + 32,
    ... < e. Units (h, a, row tile of 64 grouped rows) h-major, chunk (h*MB + a, a, h, rt);
    cost 1 + tiles, the same longest-processing-time rule on at most 4 * num_sms CTAs
    (max(units, 1) when smaller); grid = CTAs, 0 without units; aux0 = descriptors,
    aux1 = tiles, tile field 64.
  * paged prefill (variant 3): per request a descriptor (first query token, query tokens,
    first tile, end tile, L_b - qo_len_b); the request's keys [0, L_b) split into tiles
    (t, e, page, first slot) of at most 32 keys that never cross a page; units (b, kv head,
    row tile of 64 grouped rows) b-major, chunk (b, b, h, rt), cost 1 + tiles, the
    variable-block assignment rule; aux0 = descriptors, aux1 = tiles.
  * tensor-core list plans (variable blocks: variant 4 when head_dim == 128 and g in {2, 4};
    paged prefill: variant 5 when also page_size in {8, 16, 32, 64, 128}): keys in steps of
    at most 128 (variable blocks: each maximal run [s, e) of visible column blocks of (h, a)
    cut into (t, min(t + 128, e)), 2 words; paged prefill: request b's keys [0, L_b) cut into
    (t, min(t + 128, L_b)) followed by the 128 / page_size page ids kv_indices[kv_indptr[b] +
    (t + k page_size) / page_size] for t + k page_size < the step's end, else -1). Units are
    64-token row tiles: descriptor (first query token, valid tokens <= 64, first step, end
    step, key limit), with key limit = (first token + L - qo_len) for variable blocks (first
    token global) and (64 rt + L_b - qo_len_b) for paged prefill; with causal the end step is
    the first step of the row range's list whose start exceeds key limit + valid - 1 (all
    steps without causal). Variable blocks: descriptors per (h, a, rt) in that order, one
    unit (desc, 0, h, 0) each; paged prefill: descriptors per (b, rt), units (desc, 0, h, 0)
    for h = 0 .. Hkv - 1. Cost: 1 without steps, else 2 + sum over steps of 4 (more than 64
    keys) or 3; longest processing time first on at most num_sms CTAs; tile field 64;
    aux0 = descriptors, aux1 = steps.
  * paged MLA: one unit per request, len = its length from the page table (as for
    decode), tile 128, max_workers = max(1, num_sms // 2), grid = 2 P, aux0 = kv_indptr,
    aux1 = kv_indices, variant 1.

BSR (longest processing time first). Tensor-core variant (variant 1) when R == 64,
C == 64, head_dim == 128 and R*g in {128, 256} (g = Hq/Hkv): one unit per (row block
i, kv head h), rows_per_unit = R*g, at most num_sms CTAs. Otherwise the general
variant 0: rows_per_unit = 64, row_tiles = ceil(R*g / 64) units per (i, h), at most
4*num_sms CTAs. Unit u = (i*Hkv + h)*row_tiles + rt. With n = blocks in row i, cost_u =
2 + 4*(n // 2) + 3*(n % 2) for a tensor-core unit with n > 0 (1 when n == 0), and 1 + n
for a general unit. A plan for runs with a per-block token mask follows the same
rule.
Units sorted by cost descending (stable); each goes to the CTA of least current load
(ties: lowest CTA index). Chunks list each CTA's units in assignment order as
(u, i, h, rt); tile = rows_per_unit; grid = number of CTAs; aux0 = indptr,
aux1 = indices; no slots or merges.
"""

import heapq

MAGIC = 0x766B7362


def _align4(n):
    return (n + 3) & ~3


def _assemble(kind, units, worker_ptr, chunks, slots, merges, tile, aux0, aux1, grid, variant):
    off_workers = 16
    off = _align4(off_workers + len(worker_ptr))
    off_chunks = off
    off = _align4(off + 4 * len(chunks))
    off_merges = off
    off = _align4(off + 3 * len(merges))
    off_aux0 = off
    off = _align4(off + len(aux0))
    off_aux1 = off
    off = _align4(off + len(aux1))
    m = [0] * off
    hdr = [MAGIC, kind, units, max(len(worker_ptr) - 1, 0), len(chunks), slots, len(merges),
           tile, off_workers, off_chunks, off_merges, off_aux0, off_aux1, grid, off, variant]
    m[:16] = hdr
    m[off_workers:off_workers + len(worker_ptr)] = worker_ptr
    for i, c in enumerate(chunks):
        m[off_chunks + 4 * i:off_chunks + 4 * i + 4] = list(c)
    for i, it in enumerate(merges):
        m[off_merges + 3 * i:off_merges + 3 * i + 3] = list(it)
    m[off_aux0:off_aux0 + len(aux0)] = list(aux0)
    m[off_aux1:off_aux1 + len(aux1)] = list(aux1)
    return m


def linear_partition(unit_len, tile, max_workers):
    tiles = [(L + tile - 1) // tile for L in unit_len]
    starts = [0]
    for t in tiles:
        starts.append(starts[-1] + t)
    NT = starts[-1]
    P = min(max_workers, NT)
    worker_ptr, chunks = [], []
    u = 0
    for w in range(P):
        t0, t1 = (w * NT) // P, ((w + 1) * NT) // P
        worker_ptr.append(len(chunks))
        t = t0
        while t < t1:
            while starts[u + 1] <= t:
                u += 1
            e = min(t1, starts[u + 1])
            chunks.append([u, (t - starts[u]) * tile, min((e - starts[u]) * tile, unit_len[u]), -1])
            t = e
    worker_ptr.append(len(chunks))
    count = [0] * len(unit_len)
    for c in chunks:
        count[c[0]] += 1
    first = [-1] * len(unit_len)
    slots = 0
    for c in chunks:
        if count[c[0]] >= 2:
            if first[c[0]] < 0:
                first[c[0]] = slots
            c[3] = slots
            slots += 1
    merges = [(u, first[u], count[u]) for u in range(len(unit_len)) if count[u] != 1]
    return worker_ptr, chunks, slots, merges


def _slots_and_merges(unit_len, chunks):
    count = [0] * len(unit_len)
    for c in chunks:
        count[c[0]] += 1
    first = [-1] * len(unit_len)
    slots = 0
    for c in chunks:
        if count[c[0]] >= 2:
            if first[c[0]] < 0:
                first[c[0]] = slots
            c[3] = slots
            slots += 1
    merges = [(u, first[u], count[u]) for u in range(len(unit_len)) if count[u] != 1]
    return slots, merges


def _fill(tiles, T, bc, record=None):
    """Greedy left-to-right fill: a worker takes tiles while its cost stays within T. Its
    cost is its tiles plus, with bc = (pub, merge, whole): `whole` for every chunk after its
    first; `merge` once it holds two chunks and its first is the tail piece of a unit begun
    by an earlier worker (that piece is walked last, and its merge lands at the worker's
    end); `pub` for a last chunk that is the head piece of a unit continued by a later worker
    (walked first and published mid-stream). Returns the number of workers; with `record`,
    appends each worker's chunks as (unit, first tile, end tile) tuples."""
    pub, merge, whole = bc
    U = len(tiles)
    u, off, workers = 0, 0, 0
    while u < U and tiles[u] == 0:
        u += 1
    while u < U:
        workers += 1
        cost, n = 0, 0
        first_tail = off > 0
        mine = []
        while u < U:
            if tiles[u] == 0:
                u += 1
                continue
            add = 0 if n == 0 else whole + (merge if n == 1 and first_tail else 0)
            rem = tiles[u] - off
            if cost + add + rem <= T:
                mine.append((u, off, tiles[u]))
                cost += add + rem
                n += 1
                u, off = u + 1, 0
                continue
            take = T - cost - add - (pub if n > 0 else 0)
            if take > 0:
                mine.append((u, off, off + take))
                off += take
                n += 1
            break
        if record is not None:
            record.append(mine)
    return workers


def linear_partition_cost(unit_len, tile, max_workers, bc):
    """Contiguous partition of the unit tile sequence with the worker cost of _fill: the
    smallest cost bound T whose greedy fill needs at most max_workers workers, each worker
    filled up to T."""
    tiles = [(L + tile - 1) // tile for L in unit_len]
    NT = sum(tiles)
    if NT == 0:
        return linear_partition(unit_len, tile, max_workers)
    lo = max(1, -(-NT // max_workers))
    hi = NT + sum(bc) * (len(tiles) + 1)
    while lo < hi:
        mid = (lo + hi) // 2
        if _fill(tiles, mid, bc) <= max_workers:
            hi = mid
        else:
            lo = mid + 1
    rec = []
    _fill(tiles, lo, bc, rec)
    worker_ptr, chunks = [], []
    for mine in rec:
        worker_ptr.append(len(chunks))
        for u, a, b in mine:
            chunks.append([u, a * tile, min(b * tile, int(unit_len[u])), -1])
    worker_ptr.append(len(chunks))
    slots, merges = _slots_and_merges(unit_len, chunks)
    return worker_ptr, chunks, slots, merges


def decode_group_heads(num_kv_heads, page_size):
    """kv heads per unit of the page-major decode variant (0: the variant does not apply)."""
    if page_size > 16:
        return 0
    if num_kv_heads <= 8:
        return num_kv_heads
    return 8 if num_kv_heads % 8 == 0 else 0


def decode_units(kv_indptr, kv_last_page_len, batch, page_size, num_kv_heads):
    """Token count of every decode unit, in unit order."""
    G = decode_group_heads(num_kv_heads, page_size)
    per_request = num_kv_heads // G if G else num_kv_heads
    lens = []
    for b in range(batch):
        n = int(kv_indptr[b + 1]) - int(kv_indptr[b])
        L = 0 if n == 0 else (n - 1) * page_size + int(kv_last_page_len[b])
        lens += [L] * per_request
    return lens


# page-major decode: a worker's extra costs in 16-token tiles (pub, merge, whole): a piece
# published mid-stream, a merge at the worker's end, a whole-unit boundary
DECODE_BOUNDARY_TILES = (2, 2, 0)


def decode_meta(kv_indptr, kv_indices, kv_last_page_len, batch, page_size, num_qo_heads,
                num_kv_heads, num_sms, max_workers=0):
    G = decode_group_heads(num_kv_heads, page_size)
    lens = decode_units(kv_indptr, kv_last_page_len, batch, page_size, num_kv_heads)
    cap = max_workers if max_workers > 0 else (num_sms if G else 8 * num_sms)
    if G:
        wp, ch, slots, merges = linear_partition_cost(lens, 16, cap, DECODE_BOUNDARY_TILES)
    else:
        wp, ch, slots, merges = linear_partition(lens, 16, cap)
    P = len(wp) - 1
    nnz = int(kv_indptr[batch]) if batch > 0 else 0
    aux0 = [int(x) for x in kv_indptr[:batch + 1]] if batch > 0 else []
    aux1 = [int(x) for x in kv_indices[:nnz]]
    grid = P if G else (P + 7) // 8
    m = _assemble(1, len(lens), wp, ch, slots, merges, 16, aux0, aux1, grid, 1 if G else 0)
    if G:
        upb = num_kv_heads // G
        for w in range(P):
            rec = [0] * 16
            if wp[w + 1] > wp[w]:
                c = ch[wp[w + 1] - 1 if wp[w + 1] - wp[w] >= 2 else wp[w]]
                b = c[0] // upb
                pbase, npages = aux0[b], aux0[b + 1] - aux0[b]
                first = c[1] // page_size
                n = min(8, npages - first)
                rec[:7] = [c[0], c[1], c[2], c[3], pbase, npages, n]
                rec[8:8 + n] = aux1[pbase + first:pbase + first + n]
            m += rec
        m[14] = len(m)
    return m


MLA_SPLIT_PENALTY_TILES = 7


def mla_partition(unit_len, tile, max_workers):
    """Whole units by longest processing time when the busiest worker's tiles stay within
    MLA_SPLIT_PENALTY_TILES of the linear split partition's, else the linear partition."""
    tiles = [(L + tile - 1) // tile for L in unit_len]
    NT = sum(tiles)
    lin = linear_partition(unit_len, tile, max_workers)
    if NT == 0:
        return lin
    P = min(max_workers, NT)
    split_max = -(-NT // P)
    live = [u for u in range(len(unit_len)) if tiles[u] > 0]
    G = min(max_workers, len(live))
    order = sorted(range(len(live)), key=lambda i: -tiles[live[i]])   # stable
    heap = [(0, w) for w in range(G)]
    heapq.heapify(heap)
    lists = [[] for _ in range(G)]
    for i in order:
        load, w = heapq.heappop(heap)
        lists[w].append(i)
        heapq.heappush(heap, (load + tiles[live[i]], w))
    whole_max = max(sum(tiles[live[i]] for i in l) for l in lists)
    if whole_max > split_max + MLA_SPLIT_PENALTY_TILES:
        return lin
    wp, ch = [], []
    for w in range(G):
        wp.append(len(ch))
        for i in lists[w]:
            u = live[i]
            ch.append([u, 0, int(unit_len[u]), -1])
    wp.append(len(ch))
    merges = [[u, -1, 0] for u in range(len(unit_len)) if tiles[u] == 0]
    return wp, ch, 0, merges


def mla_meta(seq_lens, batch, q_len, num_sms):
    lens = []
    for b in range(batch):
        lens += [int(seq_lens[b])] * q_len
    wp, ch, slots, merges = mla_partition(lens, 128, max(1, num_sms // 2))
    return _assemble(3, len(lens), wp, ch, slots, merges, 128, [], [], 2 * (len(wp) - 1), 0)


def mla_paged_meta(kv_indptr, kv_indices, kv_last_page_len, batch, page_size, num_sms):
    lens = [paged_request_len(kv_indptr, kv_last_page_len, page_size, b) for b in range(batch)]
    wp, ch, slots, merges = mla_partition(lens, 128, max(1, num_sms // 2))
    nnz = int(kv_indptr[batch]) if batch > 0 else 0
    aux0 = [int(x) for x in kv_indptr[:batch + 1]] if batch > 0 else []
    aux1 = [int(x) for x in kv_indices[:nnz]]
    return _assemble(3, len(lens), wp, ch, slots, merges, 128, aux0, aux1, 2 * (len(wp) - 1), 1)


def paged_request_len(kv_indptr, kv_last_page_len, page_size, b):
    n = int(kv_indptr[b + 1]) - int(kv_indptr[b])
    return 0 if n == 0 else (n - 1) * page_size + int(kv_last_page_len[b])


def bsr_meta(indptr, indices, M, N, R, C, num_qo_heads, num_kv_heads, head_dim, num_sms):
    MB = (M + R - 1) // R
    g = num_qo_heads // num_kv_heads
    tc = R == 64 and C == 64 and head_dim == 128 and R * g in (128, 256)
    rows = R * g if tc else 64
    rt_n = (R * g + rows - 1) // rows
    U = MB * num_kv_heads * rt_n
    def unit_cost(u):
        i = u // (num_kv_heads * rt_n)
        n = int(indptr[i + 1]) - int(indptr[i])
        if not tc:
            return 1 + n
        return 2 + 4 * (n // 2) + 3 * (n % 2) if n > 0 else 1

    cost = [unit_cost(u) for u in range(U)]
    order = sorted(range(U), key=lambda u: -cost[u])  # Python's sort is stable
    cap = num_sms if tc else 4 * num_sms
    G = min(cap, U)
    heap = [(0, c) for c in range(G)]
    heapq.heapify(heap)
    lists = [[] for _ in range(G)]
    for u in order:
        load, c = heapq.heappop(heap)
        lists[c].append(u)
        heapq.heappush(heap, (load + cost[u], c))
    wp, ch = [], []
    for c in range(G):
        wp.append(len(ch))
        for u in lists[c]:
            ch.append([u, u // (rt_n * num_kv_heads), (u // rt_n) % num_kv_heads, u % rt_n])
    wp.append(len(ch))
    nnz = int(indptr[MB])
    return _assemble(2, U, wp, ch, 0, [], rows, [int(x) for x in indptr[:MB + 1]],
                     [int(x) for x in indices[:nnz]], G, 1 if tc else 0)


def _tc_list_shape(head_dim, num_qo_heads, num_kv_heads):
    g = num_qo_heads // num_kv_heads
    return head_dim == 128 and g in (2, 4)


def _tc_units(desc, units, cost, steps, words, tok0, ntok, tb, te, limit_first, causal, heads):
    for r0 in range(0, ntok, 64):
        valid = min(64, ntok - r0)
        lim = limit_first + r0
        end = te
        if causal:
            end = tb
            while end < te and steps[end * words] <= lim + valid - 1:
                end += 1
        d = len(desc) // 5
        desc += [tok0 + r0, valid, tb, end, lim]
        c = 1 if end == tb else 2 + sum(
            4 if steps[t * words + 1] - steps[t * words] > 64 else 3 for t in range(tb, end))
        for h in heads:
            units.append([d, 0, h, 0])
            cost.append(c)


def _lpt_chunks(units, cost, G):
    order = sorted(range(len(units)), key=lambda u: -cost[u])
    heap = [(0, c) for c in range(G)]
    heapq.heapify(heap)
    lists = [[] for _ in range(G)]
    for u in order:
        load, c = heapq.heappop(heap)
        lists[c].append(u)
        heapq.heappush(heap, (load + cost[u], c))
    wp, ch = [], []
    for c in range(G):
        wp.append(len(ch))
        for u in lists[c]:
            ch.append(units[u])
    wp.append(len(ch))
    return wp, ch


def _tc_list_meta(desc, units, cost, steps, num_sms, variant):
    U = len(units)
    G = min(num_sms, max(U, 1))
    wp, ch = _lpt_chunks(units, cost, G)
    return _assemble(2, U, wp, ch, 0, [], 64, desc, steps, G if U > 0 else 0, variant)


def bsr_variable_meta(block_mask_map, block_row_sz, block_col_sz, num_qo_heads, num_kv_heads,
                      num_sms, head_dim=64, causal=False):
    H = num_kv_heads
    if _tc_list_shape(head_dim, num_qo_heads, num_kv_heads):
        MB, NB = len(block_row_sz[0]), len(block_col_sz[0])
        qo_len = sum(int(x) for x in block_row_sz[0])
        kv_len = sum(int(x) for x in block_col_sz[0])
        steps, desc, units, cost = [], [], [], []
        for h in range(H):
            cstart, acc = [], 0
            for c in range(NB):
                cstart.append(acc)
                acc += int(block_col_sz[h][c])
            row = 0
            for a in range(MB):
                tb = len(steps) // 2
                c = 0
                while c < NB:
                    if not block_mask_map[h][a][c]:
                        c += 1
                        continue
                    s0 = cstart[c]
                    e = s0
                    while c < NB and block_mask_map[h][a][c]:
                        e += int(block_col_sz[h][c])
                        c += 1
                    for t in range(s0, e, 128):
                        steps += [t, min(t + 128, e)]
                nrow = int(block_row_sz[h][a])
                _tc_units(desc, units, cost, steps, 2, row, nrow, tb, len(steps) // 2,
                          row + kv_len - qo_len, causal, [h])
                row += nrow
        return _tc_list_meta(desc, units, cost, steps, num_sms, 4)
    g = num_qo_heads // num_kv_heads
    MB = len(block_row_sz[0])
    NB = len(block_col_sz[0])
    desc, tiles = [], []
    for h in range(H):
        cstart, acc = [], 0
        for c in range(NB):
            cstart.append(acc)
            acc += int(block_col_sz[h][c])
        row = 0
        for a in range(MB):
            nrow = int(block_row_sz[h][a])
            tb = len(tiles) // 2
            c = 0
            while c < NB:
                if not block_mask_map[h][a][c]:
                    c += 1
                    continue
                s0 = cstart[c]
                e = s0
                while c < NB and block_mask_map[h][a][c]:
                    e += int(block_col_sz[h][c])
                    c += 1
                for t in range(s0, e, 32):
                    tiles += [t, e]
            desc += [row, nrow, tb, len(tiles) // 2]
            row += nrow
    units, cost = [], []
    for h in range(H):
        for a in range(MB):
            d = (h * MB + a) * 4
            for rt in range((desc[d + 1] * g + 63) // 64):
                units.append([h * MB + a, a, h, rt])
                cost.append(1 + desc[d + 3] - desc[d + 2])
    U = len(units)
    order = sorted(range(U), key=lambda u: -cost[u])
    G = min(4 * num_sms, max(U, 1))
    heap = [(0, c) for c in range(G)]
    heapq.heapify(heap)
    lists = [[] for _ in range(G)]
    for u in order:
        load, c = heapq.heappop(heap)
        lists[c].append(u)
        heapq.heappush(heap, (load + cost[u], c))
    wp, ch = [], []
    for c in range(G):
        wp.append(len(ch))
        for u in lists[c]:
            ch.append(units[u])
    wp.append(len(ch))
    return _assemble(2, U, wp, ch, 0, [], 64, desc, tiles, G if U > 0 else 0, 2)


def prefill_paged_meta(qo_indptr, kv_indptr, kv_indices, kv_last_page_len, page_size,
                       num_qo_heads, num_kv_heads, num_sms, head_dim=64, causal=True):
    batch = len(qo_indptr) - 1
    g = num_qo_heads // num_kv_heads
    if _tc_list_shape(head_dim, num_qo_heads, num_kv_heads) and page_size in (8, 16, 32, 64, 128):
        ppk = 128 // page_size
        words = 2 + ppk
        steps, desc, units, cost = [], [], [], []
        for b in range(batch):
            nq = int(qo_indptr[b + 1]) - int(qo_indptr[b])
            L = paged_request_len(kv_indptr, kv_last_page_len, page_size, b)
            tb = len(steps) // words
            for t in range(0, L, 128):
                e = min(t + 128, L)
                steps += [t, e]
                for k in range(ppk):
                    k0 = t + k * page_size
                    steps.append(int(kv_indices[int(kv_indptr[b]) + k0 // page_size]) if k0 < e else -1)
            _tc_units(desc, units, cost, steps, words, int(qo_indptr[b]), nq, tb,
                      len(steps) // words, L - nq, causal, list(range(num_kv_heads)))
        return _tc_list_meta(desc, units, cost, steps, num_sms, 5)
    desc, tiles = [], []
    for b in range(batch):
        nq = int(qo_indptr[b + 1]) - int(qo_indptr[b])
        L = paged_request_len(kv_indptr, kv_last_page_len, page_size, b)
        tb = len(tiles) // 4
        t = 0
        while t < L:
            pi = t // page_size
            e = min(t + 32, (pi + 1) * page_size, L)
            tiles += [t, e, int(kv_indices[int(kv_indptr[b]) + pi]), t - pi * page_size]
            t = e
        desc += [int(qo_indptr[b]), nq, tb, len(tiles) // 4, L - nq]
    units, cost = [], []
    for b in range(batch):
        d = b * 5
        for h in range(num_kv_heads):
            for rt in range((desc[d + 1] * g + 63) // 64):
                units.append([b, b, h, rt])
                cost.append(1 + desc[d + 3] - desc[d + 2])
    U = len(units)
    order = sorted(range(U), key=lambda u: -cost[u])
    G = min(4 * num_sms, max(U, 1))
    heap = [(0, c) for c in range(G)]
    heapq.heapify(heap)
    lists = [[] for _ in range(G)]
    for u in order:
        load, c = heapq.heappop(heap)
        lists[c].append(u)
        heapq.heappush(heap, (load + cost[u], c))
    wp, ch = [], []
    for c in range(G):
        wp.append(len(ch))
        for u in lists[c]:
            ch.append(units[u])
    wp.append(len(ch))
    return _assemble(2, U, wp, ch, 0, [], 64, desc, tiles, G if U > 0 else 0, 3)


def sections(meta):
    """Split metadata words into a dict of named sections (for invariant checks)."""
    h = meta[:16]
    P, NC, NM = h[3], h[4], h[6]
    return dict(
        kind=h[1], units=h[2], workers=P, chunks_n=NC, slots=h[5], merges_n=NM, tile=h[7],
        grid=h[13], total=h[14], variant=h[15],
        worker_ptr=meta[h[8]:h[8] + P + 1] if P > 0 else meta[h[8]:h[8] + 1],
        chunks=[meta[h[9] + 4 * i:h[9] + 4 * i + 4] for i in range(NC)],
        merges=[meta[h[10] + 3 * i:h[10] + 3 * i + 3] for i in range(NM)],
    )
