// A small JSON reader shared by the compiler's JSON front-ends (the
// JSON-schema subset and structural tags): values keep number text as
// written, strings decoded to UTF-8; syntax errors raise CompileError
// (CG_E_SYNTAX), lone surrogates CG_E_UNSUPPORTED.
#pragma once

#include <cctype>
#include <string>
#include <utility>
#include <vector>

#include "../../../include/cg.h"
#include "ir.h"

namespace cg {

[[noreturn]] inline void json_fail(int code, const std::string& m) { throw CompileError{code, m}; }

struct JVal {
  enum T { Null, Bool, Num, Str, Arr, Obj } t = Null;
  bool b = false;
  std::string text;  // Num: source text; Str: decoded UTF-8
  std::vector<JVal> arr;
  std::vector<std::pair<std::string, JVal>> obj;

  const JVal* get(const std::string& k) const {
    const JVal* r = nullptr;
    for (auto& kv : obj) if (kv.first == k) r = &kv.second;  // last duplicate wins
    return r;
  }
  bool is_int_num() const {
    return t == Num && text.find_first_of(".eE") == std::string::npos;
  }
};

class JsonReader {
 public:
  explicit JsonReader(const std::string& s) : s_(s) {}
  explicit JsonReader(std::string&&) = delete;  // the reader keeps a reference: no temporaries
  JVal document() {
    JVal v = value();
    ws();
    if (i_ != s_.size()) json_fail(CG_E_SYNTAX, "json: trailing characters");
    return v;
  }

 private:
  const std::string& s_;
  size_t i_ = 0;

  void ws() { while (i_ < s_.size() && (s_[i_] == ' ' || s_[i_] == '\t' || s_[i_] == '\n' || s_[i_] == '\r')) ++i_; }
  bool eat(char c) { ws(); if (i_ < s_.size() && s_[i_] == c) { ++i_; return true; } return false; }
  void expect(char c) { if (!eat(c)) json_fail(CG_E_SYNTAX, std::string("json: expected '") + c + "'"); }

  static void put_utf8(std::string& o, uint32_t cp) {
    if (cp < 0x80) o.push_back(char(cp));
    else if (cp < 0x800) { o.push_back(char(0xC0 | (cp >> 6))); o.push_back(char(0x80 | (cp & 63))); }
    else if (cp < 0x10000) {
      o.push_back(char(0xE0 | (cp >> 12))); o.push_back(char(0x80 | ((cp >> 6) & 63)));
      o.push_back(char(0x80 | (cp & 63)));
    } else {
      o.push_back(char(0xF0 | (cp >> 18))); o.push_back(char(0x80 | ((cp >> 12) & 63)));
      o.push_back(char(0x80 | ((cp >> 6) & 63))); o.push_back(char(0x80 | (cp & 63)));
    }
  }
  uint32_t hex4() {
    if (i_ + 4 > s_.size()) json_fail(CG_E_SYNTAX, "json: short \\u escape");
    uint32_t v = 0;
    for (int k = 0; k < 4; ++k) {
      char c = s_[i_++];
      v <<= 4;
      if (c >= '0' && c <= '9') v |= c - '0';
      else if (c >= 'a' && c <= 'f') v |= c - 'a' + 10;
      else if (c >= 'A' && c <= 'F') v |= c - 'A' + 10;
      else json_fail(CG_E_SYNTAX, "json: bad \\u escape");
    }
    return v;
  }
  std::string string() {
    ws();
    if (i_ >= s_.size() || s_[i_] != '"') json_fail(CG_E_SYNTAX, "json: expected string");
    ++i_;
    std::string o;
    for (;;) {
      if (i_ >= s_.size()) json_fail(CG_E_SYNTAX, "json: unterminated string");
      unsigned char c = s_[i_++];
      if (c == '"') break;
      if (c < 0x20) json_fail(CG_E_SYNTAX, "json: control character in string");
      if (c != '\\') { o.push_back(char(c)); continue; }
      if (i_ >= s_.size()) json_fail(CG_E_SYNTAX, "json: dangling escape");
      char e = s_[i_++];
      switch (e) {
        case '"': o.push_back('"'); break;
        case '\\': o.push_back('\\'); break;
        case '/': o.push_back('/'); break;
        case 'b': o.push_back('\b'); break;
        case 'f': o.push_back('\f'); break;
        case 'n': o.push_back('\n'); break;
        case 'r': o.push_back('\r'); break;
        case 't': o.push_back('\t'); break;
        case 'u': {
          uint32_t cp = hex4();
          if (cp >= 0xD800 && cp < 0xDC00 && i_ + 6 <= s_.size() && s_[i_] == '\\' && s_[i_ + 1] == 'u') {
            size_t save = i_;
            i_ += 2;
            uint32_t lo = hex4();
            if (lo >= 0xDC00 && lo < 0xE000) cp = 0x10000 + ((cp - 0xD800) << 10) + (lo - 0xDC00);
            else i_ = save;
          }
          if (cp >= 0xD800 && cp < 0xE000) json_fail(CG_E_UNSUPPORTED, "lone surrogate in schema string");
          put_utf8(o, cp);
          break;
        }
        default: json_fail(CG_E_SYNTAX, "json: bad escape");
      }
    }
    return o;
  }
  JVal value() {
    ws();
    if (i_ >= s_.size()) json_fail(CG_E_SYNTAX, "json: unexpected end");
    JVal v;
    char c = s_[i_];
    if (c == '{') {
      ++i_;
      v.t = JVal::Obj;
      if (eat('}')) return v;
      do {
        std::string k = string();
        expect(':');
        v.obj.emplace_back(k, value());
      } while (eat(','));
      expect('}');
    } else if (c == '[') {
      ++i_;
      v.t = JVal::Arr;
      if (eat(']')) return v;
      do { v.arr.push_back(value()); } while (eat(','));
      expect(']');
    } else if (c == '"') {
      v.t = JVal::Str;
      v.text = string();
    } else if (s_.compare(i_, 4, "true") == 0) { v.t = JVal::Bool; v.b = true; i_ += 4; }
    else if (s_.compare(i_, 5, "false") == 0) { v.t = JVal::Bool; v.b = false; i_ += 5; }
    else if (s_.compare(i_, 4, "null") == 0) { v.t = JVal::Null; i_ += 4; }
    else if (c == '-' || (c >= '0' && c <= '9')) {
      size_t j = i_;
      if (s_[j] == '-') ++j;
      if (j >= s_.size() || !isdigit((unsigned char)s_[j])) json_fail(CG_E_SYNTAX, "json: bad number");
      if (s_[j] == '0') ++j; else while (j < s_.size() && isdigit((unsigned char)s_[j])) ++j;
      if (j < s_.size() && s_[j] == '.') {
        ++j;
        if (j >= s_.size() || !isdigit((unsigned char)s_[j])) json_fail(CG_E_SYNTAX, "json: bad number");
        while (j < s_.size() && isdigit((unsigned char)s_[j])) ++j;
      }
      if (j < s_.size() && (s_[j] == 'e' || s_[j] == 'E')) {
        ++j;
        if (j < s_.size() && (s_[j] == '+' || s_[j] == '-')) ++j;
        if (j >= s_.size() || !isdigit((unsigned char)s_[j])) json_fail(CG_E_SYNTAX, "json: bad number");
        while (j < s_.size() && isdigit((unsigned char)s_[j])) ++j;
      }
      v.t = JVal::Num;
      v.text = s_.substr(i_, j - i_);
      i_ = j;
    } else {
      json_fail(CG_E_SYNTAX, "json: unexpected character");
    }
    return v;
  }
};


int lower_json_schema_value(IR& ir, const JVal& schema, uint32_t ws_max, uint32_t max_len_default,
                            uint32_t max_items_default);

}  // namespace cg
