// pp_driver.cpp - the session driver: host bookkeeping on either side of pp_step.
//
//  * Admission and recycle: a session takes the lowest free slot and frees it on close
//    (Recipe, Notes: a recycled slot is bit-exact with a fresh engine).
//  * Prefill: voice prompt, silence, persona text, silence, then live (mhpq, "Persona
//    Voice 注入": voice + 2 x silence + persona).  During the voice and silence ticks
//    the agent's audio rows are forced; during the persona ticks the text row takes the
//    persona tokens and the audio rows are forced to silence.
//  * Acoustic delay (mhpq 3.3: 80 ms frame + 80 ms acoustic delay): in the model's
//    columns, the acoustic codebooks 1..7 of an 8-code stream are one frame behind its
//    semantic codebook 0 and the text token.  The driver takes and returns ALIGNED
//    frames (all 8 codes of one 80 ms frame together) and does the shifting:
//      user rows of tick t   = [U_t[0], U_{t-1}[1..7]]
//      agent frame f         = (text and codebook 0 of tick f, codebooks 1..7 of tick f+1)
//    with the initial token (audio_card) standing in for frame -1.  Forced agent frames
//    are shifted the same way.
#include <stdint.h>
#include <string.h>

#include <new>
#include <vector>

#include "../../include/pp.h"

namespace {

constexpr int kRows = PP_ROWS;
constexpr int kCodes = PP_USER_ROWS;   // codes of one stream's frame

struct Slot {
  int open = 0;
  int64_t tick = 0;                 // ticks run since open
  std::vector<int32_t> voice;       // [n_voice][8] aligned frames
  std::vector<int32_t> persona;     // persona text tokens
  int32_t silence[kCodes];
  int silence_ticks = 0;
  int32_t prev_col[kRows];          // the previous tick's column, model layout
  int32_t prev_user[kCodes];        // the previous aligned user frame
  int32_t pend[2];                  // text and codebook 0 of the frame still open
  int has_pend = 0;
};

}  // namespace

struct pp_driver {
  int B = 0, text_vocab = 0, audio_card = 0;
  std::vector<Slot> slots;
};

namespace {

void initial_column(const pp_driver* d, int32_t* col) {
  col[0] = d->text_vocab;
  for (int r = 1; r < kRows; ++r) col[r] = d->audio_card;
}

// The prefill phase of session tick t and, where it forces the agent, the aligned frame
// it forces (NULL when the agent's audio is free) and the forced text token (-1: free).
int phase_of(const pp_driver* d, const Slot& s, int64_t t, const int32_t** frame,
             int32_t* text) {
  (void)d;
  *frame = nullptr;
  *text = -1;
  if (t < 0) return PP_DRV_LIVE;
  const int64_t nv = (int64_t)(s.voice.size() / kCodes), np = (int64_t)s.persona.size();
  const int64_t sil = s.silence_ticks;
  if (t < nv) {
    *frame = s.voice.data() + t * kCodes;
    return PP_DRV_VOICE;
  }
  t -= nv;
  if (t < sil) {
    *frame = s.silence;
    return PP_DRV_SILENCE;
  }
  t -= sil;
  if (t < np) {
    *frame = s.silence;
    *text = s.persona[(size_t)t];
    return PP_DRV_PERSONA;
  }
  t -= np;
  if (t < sil) {
    *frame = s.silence;
    return PP_DRV_SILENCE;
  }
  return PP_DRV_LIVE;
}

bool codes_ok(const int32_t* c, int n, int card) {
  for (int i = 0; i < n; ++i)
    if (c[i] < 0 || c[i] > card) return false;
  return true;
}

}  // namespace

extern "C" {

int pp_driver_create(int max_batch, int text_vocab, int audio_card, pp_driver** out) {
  if (!out || max_batch < 1 || text_vocab < 1 || audio_card < 1) return PP_EINVAL;
  pp_driver* d = new (std::nothrow) pp_driver;
  if (!d) return PP_EINVAL;
  d->B = max_batch;
  d->text_vocab = text_vocab;
  d->audio_card = audio_card;
  d->slots.resize((size_t)max_batch);
  *out = d;
  return PP_OK;
}

void pp_driver_destroy(pp_driver* d) { delete d; }

int pp_driver_open(pp_driver* d, pp_engine* e, const pp_prompt* prompt, int* slot_out) {
  if (!d || !prompt || !slot_out) return PP_EINVAL;
  if (prompt->n_voice < 0 || prompt->n_persona < 0 || prompt->silence_ticks < 0) return PP_EINVAL;
  if ((prompt->n_voice && !prompt->voice_frames) || (prompt->n_persona && !prompt->persona_tokens))
    return PP_EINVAL;
  if (prompt->voice_frames &&
      !codes_ok(prompt->voice_frames, prompt->n_voice * kCodes, d->audio_card))
    return PP_EINVAL;
  if (prompt->silence_frame && !codes_ok(prompt->silence_frame, kCodes, d->audio_card))
    return PP_EINVAL;
  for (int i = 0; i < prompt->n_persona; ++i)
    if (prompt->persona_tokens[i] < 0 || prompt->persona_tokens[i] > d->text_vocab)
      return PP_EINVAL;
  int slot = -1;
  for (int i = 0; i < d->B; ++i)
    if (!d->slots[(size_t)i].open) {
      slot = i;
      break;
    }
  if (slot < 0) return PP_E_BUSY;
  if (e) {
    const int rc = pp_session_open(e, slot);
    if (rc != PP_OK) return rc;
  }
  Slot& s = d->slots[(size_t)slot];
  s = Slot();
  s.open = 1;
  s.voice.assign(prompt->voice_frames, prompt->voice_frames + (size_t)prompt->n_voice * kCodes);
  s.persona.assign(prompt->persona_tokens, prompt->persona_tokens + prompt->n_persona);
  for (int i = 0; i < kCodes; ++i)
    s.silence[i] = prompt->silence_frame ? prompt->silence_frame[i] : d->audio_card;
  s.silence_ticks = prompt->silence_ticks;
  initial_column(d, s.prev_col);
  for (int i = 0; i < kCodes; ++i) s.prev_user[i] = d->audio_card;
  *slot_out = slot;
  return PP_OK;
}

int pp_driver_close(pp_driver* d, pp_engine* e, int slot) {
  if (!d) return PP_EINVAL;
  if (slot < 0 || slot >= d->B) return PP_E_RANGE;
  if (!d->slots[(size_t)slot].open) return PP_E_NOTLIVE;
  if (e) {
    const int rc = pp_session_close(e, slot);
    if (rc != PP_OK) return rc;
  }
  d->slots[(size_t)slot] = Slot();
  return PP_OK;
}

int pp_driver_phase(const pp_driver* d, int slot) {
  if (!d) return PP_EINVAL;
  if (slot < 0 || slot >= d->B) return PP_E_RANGE;
  const Slot& s = d->slots[(size_t)slot];
  if (!s.open) return PP_DRV_FREE;
  const int32_t* f;
  int32_t txt;
  return phase_of(d, s, s.tick, &f, &txt);
}

int pp_driver_prepare(pp_driver* d, const int32_t* user_frames, int32_t* prev_column,
                      int32_t* user_codes, uint8_t* force_mask, int32_t* forced) {
  if (!d || !user_frames || !prev_column || !user_codes || !force_mask || !forced) return PP_EINVAL;
  for (int b = 0; b < d->B; ++b) {
    Slot& s = d->slots[(size_t)b];
    int32_t* pc = prev_column + (size_t)b * kRows;
    int32_t* uc = user_codes + (size_t)b * kCodes;
    uint8_t* fm = force_mask + (size_t)b * kRows;
    int32_t* ft = forced + (size_t)b * kRows;
    memset(fm, 0, kRows);
    memset(ft, 0, sizeof(int32_t) * kRows);
    if (!s.open) {   // the engine ignores a closed slot's inputs
      initial_column(d, pc);
      for (int i = 0; i < kCodes; ++i) uc[i] = d->audio_card;
      continue;
    }
    const int32_t* u = user_frames + (size_t)b * kCodes;
    if (!codes_ok(u, kCodes, d->audio_card)) return PP_EINVAL;
    memcpy(pc, s.prev_col, sizeof(int32_t) * kRows);
    uc[0] = u[0];                                       // semantic: this frame
    for (int i = 1; i < kCodes; ++i) uc[i] = s.prev_user[i];   // acoustic: one frame late
    // forcing: text row from this tick's phase; codebook 0 from frame t; codebooks 1..7
    // from frame t-1 (the frame whose acoustic codes this tick's column carries)
    const int32_t* now;
    const int32_t* before;
    int32_t txt, txt_before;
    phase_of(d, s, s.tick, &now, &txt);
    phase_of(d, s, s.tick - 1, &before, &txt_before);
    if (txt >= 0) {
      fm[0] = 1;
      ft[0] = txt;
    }
    if (now) {
      fm[1] = 1;
      ft[1] = now[0];
    }
    if (before || s.tick == 0) {
      // a session's first column carries the acoustic codes of frame -1, which does not
      // exist: they take the initial token
      for (int i = 1; i < kCodes; ++i) {
        fm[1 + i] = 1;
        ft[1 + i] = before ? before[i] : d->audio_card;
      }
    }
  }
  // the user frames become "previous" only once the tick has run (pp_driver_absorb)
  return PP_OK;
}

int pp_driver_absorb(pp_driver* d, const int32_t* user_frames, const int32_t* column,
                     int32_t* agent_frames) {
  if (!d || !user_frames || !column || !agent_frames) return PP_EINVAL;
  for (int b = 0; b < d->B; ++b) {
    Slot& s = d->slots[(size_t)b];
    int32_t* af = agent_frames + (size_t)b * (kCodes + 1);
    for (int i = 0; i <= kCodes; ++i) af[i] = -1;
    if (!s.open) continue;
    const int32_t* c = column + (size_t)b * kRows;
    if (s.has_pend) {   // the open frame is complete: its acoustic codes came now
      af[0] = s.pend[0];
      af[1] = s.pend[1];
      for (int i = 1; i < kCodes; ++i) af[1 + i] = c[1 + i];
    }
    s.pend[0] = c[0];
    s.pend[1] = c[1];
    s.has_pend = 1;
    memcpy(s.prev_col, c, sizeof(int32_t) * kRows);
    memcpy(s.prev_user, user_frames + (size_t)b * kCodes, sizeof(int32_t) * kCodes);
    ++s.tick;
  }
  return PP_OK;
}

int pp_driver_tick(pp_driver* d, pp_engine* e, const int32_t* user_frames,
                   int32_t* agent_frames, int32_t* column_out, void* stream) {
  if (!d || !e || !user_frames || !agent_frames) return PP_EINVAL;
  const size_t B = (size_t)d->B;
  std::vector<int32_t> prev(B * kRows), user(B * kCodes), forced(B * kRows), col(B * kRows);
  std::vector<uint8_t> mask(B * kRows);
  int rc = pp_driver_prepare(d, user_frames, prev.data(), user.data(), mask.data(), forced.data());
  if (rc != PP_OK) return rc;
  rc = pp_step_host(e, prev.data(), user.data(), mask.data(), forced.data(), col.data(), nullptr,
                    stream);
  if (rc != PP_OK) return rc;
  if (column_out) memcpy(column_out, col.data(), sizeof(int32_t) * B * kRows);
  return pp_driver_absorb(d, user_frames, col.data(), agent_frames);
}

}  // extern "C"
